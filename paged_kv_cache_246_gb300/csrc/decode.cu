// Split-KV paged decode (a query of one token per sequence) and the merge of
// the split partials.
//
// What is computed (xformers.py XFormersImpl.forward -> forward_decode;
// cpu_attn TorchSDPABackendImpl.forward -> forward_decode): for sequence b
// of length L (the new token already written), query position i = L - 1,
// query head h reading KV head h / qpk, keys lo <= j <= i with
// lo = max(0, i - W + 1) under a window W (else 0):
//     s_j = scale * q.k_j + slope_h * (j - i),   out = softmax(s) . V.
//
// Design (GB300): the kernel is HBM-bound (each cached K/V byte is read once
// and used for qpk query heads), so the work is organised around the loads.
//  * CTA = (split, KV head [, head group], sequence); 4 warps.  A split is a
//    run of `split_blocks` logical blocks; warp w takes blocks w, w+4, ...
//  * Each warp owns a ring of TMA stages in shared memory: one 4-D tiled TMA
//    copy brings one block's keys of this KV head (block_size rows x
//    head_size) and a second its values, both completing on the stage's
//    mbarrier.  Lane 0 refills a stage as soon as the warp is done with it, so
//    up to (4 warps x stages x 2 tiles) loads are in flight per CTA.
//  * q.k: lane (dg = lane % 8, ts = lane / 8) holds 8-element chunks dg
//    (and dg + 8) of the query heads in fp32 registers and dots them with the
//    same chunks of token ts, ts + 4, ...; three xor-shuffles finish each dot.
//  * Online softmax per warp in the log2 domain (q pre-scaled by
//    scale * log2 e), probabilities staged in shared memory, then p.V with each
//    lane owning head_size / 32 output dims of every query head.
//  * Warps merge through shared memory; a single split writes the output,
//    several splits write (o, m, l) partials that decode_combine_kernel
//    merges (flash-decoding).
#include <cuda_fp8.h>

#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace pkv {

constexpr int kDecWarps = 4;
constexpr int kDecThreads = kDecWarps * 32;
constexpr int kSub = 16;  // tokens per compute sub-tile
constexpr float kLazy = 8.f;  // reference-max slack (log2 units) before a rescale

struct DecodeArgs {
  void *out;
  const uint16_t *query;
  const int32_t *block_tables;
  const int32_t *seq_lens;
  const float *alibi;
  float *part_o;   // [B][H][max_splits][D]
  float *part_ml;  // [B][H][max_splits][2]
  int64_t num_blocks;
  int num_seqs, max_blocks_per_seq;
  int H, QPK, head_groups;  // head_groups = QPK / QT
  int BS, window, split_blocks, max_splits, stages;
  float scale_log2;  // scale * log2(e) (* k_scale for an fp8 cache)
  float v_scale;     // 1, or the fp8 cache's value scale
};

struct SeqSpan {
  int L;          // clamped length
  int lo;         // first visible key position
  int first_blk;  // logical block of lo
  int nblk;       // logical blocks lo .. L-1 touch
  int nsplit;     // splits this sequence uses (<= max_splits)
};

__device__ __forceinline__ SeqSpan seq_span(const DecodeArgs &a, int b, bool report) {
  SeqSpan s;
  int L = __ldg(a.seq_lens + b);
  const int cap = a.max_blocks_per_seq * a.BS;
  if (L < 0 || L > cap) {
    if (report) record_error(PKV_ERR_BOUNDS, b);
    L = L < 0 ? 0 : cap;
  }
  s.L = L;
  if (L == 0) {
    s.lo = s.first_blk = s.nblk = s.nsplit = 0;
    return s;
  }
  const int i = L - 1;
  s.lo = a.window > 0 ? max(0, i - a.window + 1) : 0;
  s.first_blk = s.lo / a.BS;
  s.nblk = i / a.BS - s.first_blk + 1;
  s.nsplit = (s.nblk + a.split_blocks - 1) / a.split_blocks;
  if (s.nsplit > a.max_splits) {  // seq_len above the host's max_seq_len
    if (report) record_error(PKV_ERR_BOUNDS, b);
    s.nsplit = a.max_splits;
  }
  return s;
}

template <class T>
__device__ __forceinline__ void load_chunk_f32(const uint4 &u, float (&f)[8]) {
  float2 t;
  t = T::to_f2(u.x); f[0] = t.x; f[1] = t.y;
  t = T::to_f2(u.y); f[2] = t.x; f[3] = t.y;
  t = T::to_f2(u.z); f[4] = t.x; f[5] = t.y;
  t = T::to_f2(u.w); f[6] = t.x; f[7] = t.y;
}

// Dots each lane finishes after the recursive halving of 4 * QT partials
// over 8 lanes, and the head of its f-th one (token is (dg >> 1) * 4 + ts).
template <int QT> struct NfOf { static constexpr int v = QT >= 2 ? QT / 2 : 1; };
template <int QT>
__device__ __forceinline__ int head_of(int dg, int f) {
  if constexpr (QT == 4) return 2 * (dg & 1) + f;
  else if constexpr (QT == 2) return dg & 1;
  else return 0;
}

// One halving level over lanes xor MASK: N values -> N / 2 (or a plain sum
// when one value is left).
template <int N, int MASK>
__device__ __forceinline__ void halve(float *v, int lane) {
  if constexpr (N >= 2) {
    const bool up = (lane & MASK) != 0;
#pragma unroll
    for (int k = 0; k < N / 2; ++k) {
      const float send = up ? v[k] : v[k + N / 2];
      const float keep = up ? v[k + N / 2] : v[k];
      v[k] = keep + __shfl_xor_sync(0xffffffffu, send, MASK);
    }
  } else {
    v[0] += __shfl_xor_sync(0xffffffffu, v[0], MASK);
  }
}

template <int NV>
__device__ __forceinline__ void reduce_over_dg(float *v, int lane) {
  halve<NV, 4>(v, lane);
  halve<(NV >= 2 ? NV / 2 : 1), 2>(v, lane);
  halve<(NV >= 4 ? NV / 4 : 1), 1>(v, lane);
}

// Eight / four / two E4M3 cache codes (low byte first) widened to fp32.
__device__ __forceinline__ float2 e4m3x2_to_f2(uint32_t two) {
  const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(
      static_cast<__nv_fp8x2_storage_t>(two & 0xffffu), __NV_E4M3);
  return __half22float2(*reinterpret_cast<const __half2 *>(&h));
}
__device__ __forceinline__ void load_chunk8_f32(const uint2 &u, float (&f)[8]) {
  float2 t;
  t = e4m3x2_to_f2(u.x); f[0] = t.x; f[1] = t.y;
  t = e4m3x2_to_f2(u.x >> 16); f[2] = t.x; f[3] = t.y;
  t = e4m3x2_to_f2(u.y); f[4] = t.x; f[5] = t.y;
  t = e4m3x2_to_f2(u.y >> 16); f[6] = t.x; f[7] = t.y;
}

// T: element type of queries / outputs; D: head size; QT: query heads per
// CTA (<= 4); KV8: the cache holds E4M3 codes (k_scale is folded into the
// query scale, v_scale applied to the merged output).
template <class T, int D, int QT, bool KV8>
__global__ void __launch_bounds__(kDecThreads, KV8 ? 4 : 3)
decode_split_kernel(const DecodeArgs a, const __grid_constant__ CUtensorMap tmap) {
  constexpr int CPL = D / 64;  // 8-element chunks per lane per token (q.k)
  constexpr int DPL = D / 32;  // output dims per lane (p.V)
  constexpr int ROWC = D / 8;  // 16-byte chunks per K/V row
  extern __shared__ __align__(128) uint8_t smem[];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int split = blockIdx.x;
  const int kvh = blockIdx.y / a.head_groups;
  const int hgrp = blockIdx.y % a.head_groups;
  const int b = blockIdx.z;
  const int head0 = kvh * a.QPK + hgrp * QT;  // first query head of this CTA
  const int BS = a.BS;
  const int nst = a.stages;
  const int tile_elems = BS * D;
  constexpr int EB = KV8 ? 1 : 2;  // cache bytes per element
  const uint32_t tile_bytes = static_cast<uint32_t>(tile_elems) * EB;

  const SeqSpan sp = seq_span(a, b, split == 0 && blockIdx.y == 0 && threadIdx.x == 0);
  const int H = a.H;
  if (sp.L == 0) {  // no keys: the output row is zero
    if (split == 0) {
      uint16_t *o = static_cast<uint16_t *>(a.out) + static_cast<int64_t>(b) * H * D + head0 * D;
      for (int k = threadIdx.x; k < QT * D; k += kDecThreads) o[k] = 0;
    }
    return;
  }
  const int blk_begin = sp.first_blk + split * a.split_blocks;
  const int blk_end = min(blk_begin + a.split_blocks, sp.first_blk + sp.nblk);
  if (split >= sp.nsplit || blk_begin >= blk_end) return;
  const int nb_split = blk_end - blk_begin;

  // ---- shared memory carve-up -------------------------------------------
  uint8_t *tiles = smem;  // [warp][stage][K,V][tile]
  float *sP = reinterpret_cast<float *>(smem + static_cast<size_t>(kDecWarps) * nst * 2 * tile_bytes);
  int32_t *sTable = reinterpret_cast<int32_t *>(sP + kDecWarps * kSub * QT);
  uint64_t *bars = reinterpret_cast<uint64_t *>(
      reinterpret_cast<uint8_t *>(sTable) + ((a.split_blocks * 4 + 15) / 16) * 16);

  if (threadIdx.x == 0) prefetch_tensormap(&tmap);
  // Physical blocks of this split, range-checked once.
  const int32_t *trow = a.block_tables + static_cast<int64_t>(b) * a.max_blocks_per_seq;
  for (int k = threadIdx.x; k < nb_split; k += kDecThreads) {
    int32_t pb = __ldg(trow + blk_begin + k);
    if (pb < 0 || pb >= a.num_blocks) {
      record_error(PKV_ERR_BOUNDS, static_cast<int64_t>(b) * a.max_blocks_per_seq + blk_begin + k);
      pb = 0;
    }
    sTable[k] = pb;
  }
  uint64_t *wbar = bars + warp * nst;
  if (lane == 0) {
    for (int st = 0; st < nst; ++st) mbar_init(&wbar[st], 1);
    fence_mbar_init();
  }
  __syncthreads();

  // ---- this warp's blocks: k-th is split block warp + 4k -------------------
  const int my_count = nb_split > warp ? (nb_split - warp + kDecWarps - 1) / kDecWarps : 0;
  uint8_t *wtiles = tiles + static_cast<size_t>(warp) * nst * 2 * tile_bytes;
  auto issue = [&](int k) {
    const int st = k % nst;
    const int pb = sTable[warp + k * kDecWarps];
    mbar_arrive_expect_tx(&wbar[st], 2u * tile_bytes);
    uint8_t *kt = wtiles + static_cast<size_t>(st) * 2 * tile_bytes;
    tma_load_4d(kt, &tmap, &wbar[st], 0, kvh, pb * BS, 0);
    tma_load_4d(kt + tile_bytes, &tmap, &wbar[st], 0, kvh, pb * BS, 1);
  };
  int issued = 0;
  if (lane == 0) {
    for (; issued < min(nst, my_count); ++issued) issue(issued);
  }

  // ---- query registers (pre-scaled into the log2 domain) ------------------
  const int dg = lane & 7, ts = lane >> 3;
  unsigned long long q2[QT][CPL * 4];  // packed dim pairs
  {
    const uint4 *qrow = reinterpret_cast<const uint4 *>(a.query + (static_cast<int64_t>(b) * H + head0) * D);
#pragma unroll
    for (int h = 0; h < QT; ++h)
#pragma unroll
      for (int c = 0; c < CPL; ++c) {
        float f[8];
        load_chunk_f32<T>(__ldg(qrow + h * ROWC + c * 8 + dg), f);
#pragma unroll
        for (int e = 0; e < 8; e += 2)
          q2[h][c * 4 + e / 2] = f2pack(f[e] * a.scale_log2, f[e + 1] * a.scale_log2);
      }
  }
  float slope[QT];
#pragma unroll
  for (int h = 0; h < QT; ++h) slope[h] = a.alibi ? __ldg(a.alibi + head0 + h) * kLog2e : 0.f;

  constexpr int NF = NfOf<QT>::v;  // dots (heads) each lane finishes per sub-tile
  float slope_own[NF];  // ALiBi slopes of this lane's heads head_of(dg, f)
#pragma unroll
  for (int f = 0; f < NF; ++f) {
    if constexpr (QT == 4) slope_own[f] = (dg & 1) ? slope[2 + f] : slope[f];
    else if constexpr (QT == 2) slope_own[f] = (dg & 1) ? slope[1] : slope[0];
    else slope_own[f] = slope[0];
  }
  float m[NF], l[NF];
  unsigned long long o2[QT][DPL / 2];  // packed output dim pairs
#pragma unroll
  for (int f = 0; f < NF; ++f) {
    m[f] = -INFINITY;
    l[f] = 0.f;
  }
#pragma unroll
  for (int h = 0; h < QT; ++h)
#pragma unroll
    for (int e = 0; e < DPL / 2; ++e) o2[h][e] = 0ull;  // (+0, +0)
  float *wP = sP + warp * kSub * QT;
  const int qpos = sp.L - 1;
  bool ok = true;
  int consumed = 0;

  for (int k = 0; k < my_count; ++k) {
    const int st = k % nst;
    // every lane observes the phase (acquire); the verdict is warp-uniform
    const bool got = mbar_wait_bounded(&wbar[st], (k / nst) & 1, b);
    if (!__all_sync(0xffffffffu, got)) {
      ok = false;
      break;
    }
    consumed = k + 1;
    const uint8_t *kt = wtiles + static_cast<size_t>(st) * 2 * tile_bytes;
    const uint8_t *vt = kt + tile_bytes;
    const int blk = blk_begin + warp + k * kDecWarps;  // logical block
    for (int sub = 0; sub < BS; sub += kSub) {
      const int j0 = blk * BS + sub;  // position of the sub-tile's token 0
      const int t_lo = max(sp.lo - j0, 0);
      const int t_hi = min(sp.L - j0, kSub);
      if (t_lo >= t_hi) continue;  // warp-uniform
      // ---- q.k for 16 tokens: lane (dg, ts) accumulates partial dots of
      // tokens it*4 + ts over its dims, index it * QT + h ---------------------
      constexpr int NV = (kSub / 4) * QT;  // partial dots per lane
      float v[NV];
      const uint4 *k4 = reinterpret_cast<const uint4 *>(kt + sub * D * EB);
      const uint2 *k2 = reinterpret_cast<const uint2 *>(kt + sub * D * EB);
#pragma unroll
      for (int it = 0; it < kSub / 4; ++it) {
        const int tok = it * 4 + ts;
        unsigned long long acc[QT];  // even / odd dim partial sums
#pragma unroll
        for (int h = 0; h < QT; ++h) acc[h] = 0ull;
#pragma unroll
        for (int c = 0; c < CPL; ++c) {
          float f[8];
          if constexpr (KV8)
            load_chunk8_f32(k2[tok * ROWC + c * 8 + dg], f);
          else
            load_chunk_f32<T>(k4[tok * ROWC + c * 8 + dg], f);
#pragma unroll
          for (int e = 0; e < 8; e += 2) {
            const unsigned long long kk = f2pack(f[e], f[e + 1]);
#pragma unroll
            for (int h = 0; h < QT; ++h) acc[h] = ffma2(q2[h][c * 4 + e / 2], kk, acc[h]);
          }
        }
#pragma unroll
        for (int h = 0; h < QT; ++h) {
          float x, y;
          f2unpack(acc[h], x, y);
          v[it * QT + h] = x + y;
        }
      }
      // Recursive halving over the 8 dg lanes (xor 4, 2, 1): each level a lane
      // keeps half of its values and adds the partner's copy of that half, so
      // the 8 lanes finish the NV dots between them (NF each) instead of every
      // lane finishing all of them.
      reduce_over_dg<NV>(v, lane);
      // lane now holds NF dots of token tk = (dg >> 1) * 4 + ts, heads head_of(dg, f)
      const int tk = (dg >> 1) * 4 + ts;
      const int j = j0 + tk;
      const bool valid = tk >= t_lo && tk < t_hi;
      float sc[NF];
#pragma unroll
      for (int f = 0; f < NF; ++f)
        sc[f] = valid ? v[f] + slope_own[f] * static_cast<float>(j - qpos) : -INFINITY;
      // ---- online softmax with a lazy reference max: while no score exceeds
      // the head's reference m by more than kLazy (log2 units) the weights
      // 2^(s - m) stay <= 2^kLazy and nothing is rescaled; otherwise the
      // reference moves to the true running max (the 16 lanes of a head) --
      bool grow = false;
#pragma unroll
      for (int f = 0; f < NF; ++f) grow |= sc[f] > m[f] + kLazy;
      if (!__any_sync(0xffffffffu, grow)) {
#pragma unroll
        for (int f = 0; f < NF; ++f) {
          const float p = fast_exp2(sc[f] - m[f]);
          l[f] += p;
          if (QT > 1 || (dg & 1) == 0) wP[tk * QT + head_of<QT>(dg, f)] = p;
        }
        __syncwarp();
      } else {
        float alpha_own[NF];
#pragma unroll
        for (int f = 0; f < NF; ++f) {
          float bm = sc[f];
          bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 2));
          bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 4));
          bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 8));
          bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 16));
          const float mn = fmaxf(m[f], bm);
          alpha_own[f] = fast_exp2(m[f] - mn);
          m[f] = mn;
          const float p = fast_exp2(sc[f] - mn);
          l[f] = l[f] * alpha_own[f] + p;  // per-lane partial, summed at the end
          if (QT > 1 || (dg & 1) == 0) wP[tk * QT + head_of<QT>(dg, f)] = p;
        }
        // every lane needs every head's rescale factor for its p.V accumulators
        float alpha[QT];
        if constexpr (QT == 4) {
          const float x0 = __shfl_xor_sync(0xffffffffu, alpha_own[0], 1);
          const float x1 = __shfl_xor_sync(0xffffffffu, alpha_own[1], 1);
          const bool hi = dg & 1;
          alpha[0] = hi ? x0 : alpha_own[0];
          alpha[1] = hi ? x1 : alpha_own[1];
          alpha[2] = hi ? alpha_own[0] : x0;
          alpha[3] = hi ? alpha_own[1] : x1;
        } else if constexpr (QT == 2) {
          const float x0 = __shfl_xor_sync(0xffffffffu, alpha_own[0], 1);
          const bool hi = dg & 1;
          alpha[0] = hi ? x0 : alpha_own[0];
          alpha[1] = hi ? alpha_own[0] : x0;
        } else {
          alpha[0] = alpha_own[0];
        }
#pragma unroll
        for (int h = 0; h < QT; ++h) {
          const unsigned long long a2 = f2pack(alpha[h], alpha[h]);
#pragma unroll
          for (int e = 0; e < DPL / 2; ++e) o2[h][e] = fmul2(o2[h][e], a2);
        }
        __syncwarp();
      }
      // ---- p.V over the valid tokens ---------------------------------------
      const uint8_t *vrow = vt + (sub * D + lane * DPL) * EB;
      for (int tok = t_lo; tok < t_hi; ++tok) {
        float vf[DPL];
        if constexpr (KV8 && DPL == 4) {
          const uint32_t u = *reinterpret_cast<const uint32_t *>(vrow + tok * D);
          float2 t0 = e4m3x2_to_f2(u), t1 = e4m3x2_to_f2(u >> 16);
          vf[0] = t0.x; vf[1] = t0.y; vf[2] = t1.x; vf[3] = t1.y;
        } else if constexpr (KV8) {
          const uint32_t u = *reinterpret_cast<const uint16_t *>(vrow + tok * D);
          float2 t0 = e4m3x2_to_f2(u);
          vf[0] = t0.x; vf[1] = t0.y;
        } else if constexpr (DPL == 4) {
          const uint2 u = *reinterpret_cast<const uint2 *>(vrow + tok * D * 2);
          float2 t0 = T::to_f2(u.x), t1 = T::to_f2(u.y);
          vf[0] = t0.x; vf[1] = t0.y; vf[2] = t1.x; vf[3] = t1.y;
        } else {
          const uint32_t u = *reinterpret_cast<const uint32_t *>(vrow + tok * D * 2);
          float2 t0 = T::to_f2(u);
          vf[0] = t0.x; vf[1] = t0.y;
        }
        float pp[QT];
        if constexpr (QT == 4) {
          const float4 p4 = *reinterpret_cast<const float4 *>(wP + tok * 4);
          pp[0] = p4.x; pp[1] = p4.y; pp[2] = p4.z; pp[3] = p4.w;
        } else {
#pragma unroll
          for (int h = 0; h < QT; ++h) pp[h] = wP[tok * QT + h];
        }
        unsigned long long vv[DPL / 2];
#pragma unroll
        for (int e = 0; e < DPL / 2; ++e) vv[e] = f2pack(vf[2 * e], vf[2 * e + 1]);
#pragma unroll
        for (int h = 0; h < QT; ++h) {
          const unsigned long long p2 = f2pack(pp[h], pp[h]);
#pragma unroll
          for (int e = 0; e < DPL / 2; ++e) o2[h][e] = ffma2(p2, vv[e], o2[h][e]);
        }
      }
      __syncwarp();
    }
    // stage st is free again: refill it
    if (lane == 0 && issued < my_count) {
      issue(issued);
      ++issued;
    }
    __syncwarp();
  }
  issued = __shfl_sync(0xffffffffu, issued, 0);
  if (!ok) {  // drain this warp's copies still in flight, bounded
    for (int k = consumed; k < issued; ++k) mbar_wait_bounded(&wbar[k % nst], (k / nst) & 1, b);
  }

  // ---- merge the 4 warps' softmax states ----------------------------------
  __syncthreads();  // every warp's TMA traffic has landed; tiles are reusable
  float *sM = reinterpret_cast<float *>(smem);          // [warp][QT]
  float *sL = sM + kDecWarps * QT;                       // [warp][QT]
  float *sO = sL + kDecWarps * QT;                       // [warp][QT][D]
#pragma unroll
  for (int h = 0; h < QT; ++h)
#pragma unroll
    for (int e = 0; e < DPL / 2; ++e) {
      float x, y;
      f2unpack(o2[h][e], x, y);
      sO[(warp * QT + h) * D + lane * DPL + 2 * e] = x;
      sO[(warp * QT + h) * D + lane * DPL + 2 * e + 1] = y;
    }
#pragma unroll
  for (int f = 0; f < NF; ++f) {
    float lt = l[f];
    lt += __shfl_xor_sync(0xffffffffu, lt, 2);
    lt += __shfl_xor_sync(0xffffffffu, lt, 4);
    lt += __shfl_xor_sync(0xffffffffu, lt, 8);
    lt += __shfl_xor_sync(0xffffffffu, lt, 16);
    if (lane < 2 && (QT > 1 || lane == 0)) {
      const int hf = head_of<QT>(lane, f);
      sM[warp * QT + hf] = m[f];
      sL[warp * QT + hf] = lt;
    }
  }
  __syncthreads();
  const bool single = sp.nsplit == 1;
  for (int idx = threadIdx.x; idx < QT * D; idx += kDecThreads) {
    const int h = idx / D, d = idx % D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kDecWarps; ++w) M = fmaxf(M, sM[w * QT + h]);
    float num = 0.f, den = 0.f;
#pragma unroll
    for (int w = 0; w < kDecWarps; ++w) {
      const float e = fast_exp2(sM[w * QT + h] - M);
      num = fmaf(e, sO[(w * QT + h) * D + d], num);
      den = fmaf(e, sL[w * QT + h], den);
    }
    const float val = num / den * a.v_scale;
    const int64_t hh = static_cast<int64_t>(b) * H + head0 + h;
    if (single) {
      uint16_t *o16 = static_cast<uint16_t *>(a.out);
      const uint32_t packed = T::from_f2(val, 0.f);
      o16[hh * D + d] = static_cast<uint16_t>(packed & 0xffffu);
    } else {
      const int64_t slot = hh * a.max_splits + split;
      a.part_o[slot * D + d] = val;
      if (d == 0) {
        a.part_ml[slot * 2] = M;
        a.part_ml[slot * 2 + 1] = den;
      }
    }
  }
}

// One CTA per (query head, sequence) with more than one split.
template <class T, int D>
__global__ void __launch_bounds__(D) decode_combine_kernel(const DecodeArgs a) {
  const int h = blockIdx.x, b = blockIdx.y;
  const SeqSpan sp = seq_span(a, b, false);
  if (sp.nsplit <= 1) return;  // the split kernel wrote the output itself
  const int64_t hh = static_cast<int64_t>(b) * a.H + h;
  const float *ml = a.part_ml + hh * a.max_splits * 2;
  float M = -INFINITY;
  for (int s = 0; s < sp.nsplit; ++s) M = fmaxf(M, ml[2 * s]);
  const int d = threadIdx.x;
  const float *po = a.part_o + hh * a.max_splits * D + d;
  float num = 0.f, den = 0.f;
  for (int s = 0; s < sp.nsplit; ++s) {
    const float w = fast_exp2(ml[2 * s] - M) * ml[2 * s + 1];
    num = fmaf(w, po[static_cast<int64_t>(s) * D], num);
    den += w;
  }
  const float val = num / den;
  uint16_t *o16 = static_cast<uint16_t *>(a.out);
  o16[hh * D + d] = static_cast<uint16_t>(T::from_f2(val, 0.f) & 0xffffu);
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
static int stages_for(int BS) { return BS <= 16 ? 2 : 1; }

static size_t split_smem_bytes(int BS, int D, int QT, int split_blocks, int eb) {
  const size_t tiles = static_cast<size_t>(kDecWarps) * stages_for(BS) * 2 * BS * D * eb;
  const size_t p = static_cast<size_t>(kDecWarps) * kSub * QT * 4;
  const size_t table = ((split_blocks * 4 + 15) / 16) * 16;
  const size_t bars = static_cast<size_t>(kDecWarps) * stages_for(BS) * 8;
  return tiles + p + table + bars;
}

DecodePlan plan_decode(int num_seqs, int max_seq_len, const Geometry &g, int sms) {
  DecodePlan p{};
  const int BS = g.BS;
  int eff = max_seq_len;
  int eff_blocks;
  if (g.window > 0 && g.window < max_seq_len) {
    eff = g.window;
    eff_blocks = (eff + BS - 1) / BS + 1;  // a window start can straddle a block
  } else {
    eff_blocks = (eff + BS - 1) / BS;
  }
  eff_blocks = std::max(eff_blocks, 1);
  const int QT = g.QPK >= 4 ? 4 : g.QPK;
  const int64_t items = static_cast<int64_t>(num_seqs) * g.KVH * (g.QPK / QT);
  // Splits of ~1024 tokens bound the longest CTA (load balance over uneven
  // lengths) while keeping the fp32 partials small; shrink them while the
  // grid would leave SMs idle.  (Measured, 256 sequences of 512..4096 tokens:
  // 0.889 / 0.918 / 0.900 of HBM with 512 / 1024 / 2048-token splits.)
  int split_blocks = std::max(1024 / BS, 4);
  while (split_blocks > 8 &&
         items * ((eff_blocks + split_blocks - 1) / split_blocks) < 8LL * sms)
    split_blocks /= 2;
  if (eff_blocks <= 2 * split_blocks) split_blocks = eff_blocks;  // short: one split
  p.split_blocks = split_blocks;
  p.max_splits = (eff_blocks + split_blocks - 1) / split_blocks;
  p.workspace_bytes = 0;
  if (p.max_splits > 1) {
    const size_t n = static_cast<size_t>(num_seqs) * g.H * p.max_splits;
    p.workspace_bytes = n * g.D * 4 + n * 2 * 4;
    p.workspace_bytes = (p.workspace_bytes + 255) / 256 * 256;
  }
  return p;
}

template <class T, int D, int QT, bool KV8>
static cudaError_t launch_typed(const DecodeArgs &a, const CUtensorMap &tmap, int KVH, int num_seqs,
                                cudaStream_t stream) {
  const size_t smem = split_smem_bytes(a.BS, D, QT, a.split_blocks, KV8 ? 1 : 2);
  auto kern = decode_split_kernel<T, D, QT, KV8>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  dim3 grid(a.max_splits, KVH * a.head_groups, num_seqs);
  kern<<<grid, kDecThreads, smem, stream>>>(a, tmap);
  e = cudaGetLastError();
  if (e != cudaSuccess || a.max_splits <= 1) return e;
  decode_combine_kernel<T, D><<<dim3(a.H, num_seqs), D, 0, stream>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_decode(void *out, const void *query, int num_seqs, const void *kv_cache,
                          const int32_t *block_tables, int max_blocks_per_seq,
                          const int32_t *seq_lens, int max_seq_len, const Geometry &g,
                          const DecodePlan &plan, void *workspace, cudaStream_t stream) {
  (void)max_seq_len;
  // Tensor map over the whole cache: (D, KVH, NB * BS tokens, 2 halves).
  CUtensorMap tmap;
  const cuuint64_t dims[4] = {static_cast<cuuint64_t>(g.D), static_cast<cuuint64_t>(g.KVH),
                              static_cast<cuuint64_t>(g.num_blocks * g.BS), 2};
  const cuuint64_t eb = static_cast<cuuint64_t>(g.elem_bytes);
  const cuuint64_t strides[3] = {static_cast<cuuint64_t>(g.D) * eb,
                                 static_cast<cuuint64_t>(g.row_elems) * eb,
                                 static_cast<cuuint64_t>(g.num_blocks * g.block_elems) * eb};
  const cuuint32_t box[4] = {static_cast<cuuint32_t>(g.D), 1, static_cast<cuuint32_t>(g.BS), 1};
  const CUtensorMapDataType dt =
      g.fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8
            : (g.dtype == PKV_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                   : CU_TENSOR_MAP_DATA_TYPE_FLOAT16);
  if (encode_tensor_map(&tmap, dt, 4, const_cast<void *>(kv_cache), dims, strides, box,
                        CU_TENSOR_MAP_SWIZZLE_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;

  DecodeArgs a{};
  a.out = out;
  a.query = static_cast<const uint16_t *>(query);
  a.block_tables = block_tables;
  a.seq_lens = seq_lens;
  a.alibi = g.alibi;
  const size_t n = static_cast<size_t>(num_seqs) * g.H * plan.max_splits;
  a.part_o = static_cast<float *>(workspace);
  a.part_ml = plan.max_splits > 1 ? a.part_o + n * g.D : nullptr;
  a.num_blocks = g.num_blocks;
  a.num_seqs = num_seqs;
  a.max_blocks_per_seq = max_blocks_per_seq;
  a.H = g.H;
  a.QPK = g.QPK;
  const int QT = g.QPK >= 4 ? 4 : g.QPK;
  a.head_groups = g.QPK / QT;
  a.BS = g.BS;
  a.window = g.window;
  a.split_blocks = plan.split_blocks;
  a.max_splits = plan.max_splits;
  a.stages = stages_for(g.BS);
  a.scale_log2 = g.scale * kLog2e * g.k_scale;
  a.v_scale = g.v_scale;

  const bool bf = g.dtype == PKV_BF16;
#define PKV_DEC(TT, DD, QQ)                                                    \
  if (g.D == DD && QT == QQ)                                                   \
    return g.fp8 ? launch_typed<TT, DD, QQ, true>(a, tmap, g.KVH, num_seqs, stream) \
                 : launch_typed<TT, DD, QQ, false>(a, tmap, g.KVH, num_seqs, stream);
  if (bf) {
    PKV_DEC(BF16, 128, 4) PKV_DEC(BF16, 128, 2) PKV_DEC(BF16, 128, 1)
    PKV_DEC(BF16, 64, 4) PKV_DEC(BF16, 64, 2) PKV_DEC(BF16, 64, 1)
  } else {
    PKV_DEC(FP16, 128, 4) PKV_DEC(FP16, 128, 2) PKV_DEC(FP16, 128, 1)
    PKV_DEC(FP16, 64, 4) PKV_DEC(FP16, 64, 2) PKV_DEC(FP16, 64, 1)
  }
#undef PKV_DEC
  return cudaErrorInvalidValue;
}

// ---------------------------------------------------------------------------
// Static decode scratch for callers that cannot allocate device memory.
//
// The split partials of paged_attn_decode_noalloc live in this file-scope
// array instead of a caller workspace.  The array belongs to the module, so
// every GPU that loads this library holds it until the process exits.  In
// host code its name is only a host-side stand-in: the device address must be
// looked up (once per device, with that device current) and passed to the
// kernels.  All calls share the array and it keeps the last call's contents;
// nothing in it has to start at zero, because the combine pass only reads
// partials the split pass of the same call has just written.  Calls whose
// work overlaps on the GPU (different streams, or before the previous call
// has finished) race on it.
// ---------------------------------------------------------------------------
static __device__ __align__(256) unsigned char g_decode_scratch[PKV_DECODE_STATIC_SCRATCH_BYTES];

static void *g_scratch_addr[64];
static bool g_scratch_known[64];
static std::mutex g_scratch_mu;

cudaError_t static_decode_scratch(void **ptr, size_t *bytes) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (!g_scratch_known[dev]) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_decode_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = p;
    g_scratch_known[dev] = true;
  }
  *ptr = g_scratch_addr[dev];
  *bytes = sizeof(g_decode_scratch);
  return cudaSuccess;
}

cudaError_t read_device_error_decode(unsigned long long *out) {
  return read_and_clear_unit_error(out);
}

}  // namespace pkv
