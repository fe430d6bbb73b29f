// Device-side routing pieces shared by the routing kernels (route.cu) and the
// decode megakernel (decode.cu). Outputs go wherever the RouteArgs pointers
// point (global or shared memory); logits are read through L2.
#pragma once

#include <cmath>

#include "common.cuh"
#include "kernels.h"

namespace moe {

// In-place exclusive prefix sum of n ints in shared memory; returns the total.
// Called by all threads of the block. scratch: 33 ints of shared memory.
__device__ __forceinline__ int block_exclusive_scan(int* data, int n, int* scratch) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nwarps = blockDim.x >> 5;
  const int per = (n + blockDim.x - 1) / blockDim.x;
  const int start = tid * per;
  int local = 0;
  for (int i = 0; i < per; ++i) {
    const int idx = start + i;
    if (idx < n) local += data[idx];
  }
  int incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) scratch[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int wv = (lane < nwarps) ? scratch[lane] : 0;
    int wincl = wv;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, wincl, o);
      if (lane >= o) wincl += y;
    }
    scratch[lane] = wincl - wv;
    if (lane == 31) scratch[32] = wincl;
  }
  __syncthreads();
  int base = scratch[warp] + incl - local;
  for (int i = 0; i < per; ++i) {
    const int idx = start + i;
    if (idx < n) {
      const int c = data[idx];
      data[idx] = base;
      base += c;
    }
  }
  const int total = scratch[32];
  __syncthreads();
  return total;
}

// Router logits for T <= kSmallRouteMaxT tokens are summed in two fixed
// levels: kLogitParts warp partials per expert row (each a lane-strided FP32
// FMA chain over 1/kLogitParts of the row, then a butterfly), then the
// partials in order p = 0..kLogitParts-1 plus the bias. Every small-batch path
// uses these two functions, so they agree bit for bit.
constexpr int kLogitParts = 16;

// Partial p of expert e's logits for every token, written to part[t][e][p].
// TMAX: the largest T the caller passes (the token loop is unrolled to it;
// every token's FMA chain is the same whatever TMAX is).
template <int TMAX = kSmallRouteMaxT>
__device__ __forceinline__ void warp_logit_partial(const RouteArgs& a, int e, int p, float* part) {
  const int lane = threadIdx.x & 31;
  const int T = a.T, H = a.H, E = a.E;
  const int h4b = (p * (H / 4)) / kLogitParts, h4e = ((p + 1) * (H / 4)) / kLogitParts;
  float acc[TMAX];
#pragma unroll
  for (int t = 0; t < TMAX; ++t) acc[t] = 0.f;
  const float4* wr4 = reinterpret_cast<const float4*>(a.wr + (size_t)e * H) + h4b;
  const uint2* x2 = reinterpret_cast<const uint2*>(a.x) + h4b;
#pragma unroll 2
  for (int h4 = lane; h4 < h4e - h4b; h4 += 32) {
    const float4 wv = __ldg(wr4 + h4);
#pragma unroll
    for (int t = 0; t < TMAX; ++t) {
      if (t < T) {
        const uint2 raw = __ldg(x2 + (size_t)t * (H / 4) + h4);
        const float2 x01 = __half22float2(*reinterpret_cast<const __half2*>(&raw.x));
        const float2 x23 = __half22float2(*reinterpret_cast<const __half2*>(&raw.y));
        acc[t] = fmaf(wv.x, x01.x, acc[t]);
        acc[t] = fmaf(wv.y, x01.y, acc[t]);
        acc[t] = fmaf(wv.z, x23.x, acc[t]);
        acc[t] = fmaf(wv.w, x23.y, acc[t]);
      }
    }
  }
#pragma unroll
  for (int t = 0; t < TMAX; ++t)
    if (t < T) {
      const float v = warp_sum(acc[t]);
      if (lane == 0) part[((size_t)t * E + e) * kLogitParts + p] = v;
    }
}

// Logit (t, e) from its kLogitParts partials (16 consecutive floats, read
// through L2): summed in order, then the bias.
__device__ __forceinline__ float logit_from_parts(const RouteArgs& a, const float* part, int t, int e) {
  const float4* p4 = reinterpret_cast<const float4*>(part + ((size_t)t * a.E + e) * kLogitParts);
  float v = 0.f;
#pragma unroll
  for (int q = 0; q < kLogitParts / 4; ++q) {
    const float4 u = __ldcg(p4 + q);
    v += u.x;
    v += u.y;
    v += u.z;
    v += u.w;
  }
  return v + (a.bias ? __ldg(a.bias + e) : 0.f);
}

// Logit (t, e) of the large-batch path from its nsplit K-part planes
// ([p][T][E], read through L2): summed in order p = 0..nsplit-1, then the bias.
__device__ __forceinline__ float logit_from_planes(const RouteArgs& a, int t, int e) {
  const size_t plane = (size_t)a.T * a.E;
  const float* q = a.logits + (size_t)t * a.E + e;
  float u[kRouterSplitMax];
#pragma unroll
  for (int p = 0; p < kRouterSplitMax; ++p) u[p] = p < a.nsplit ? __ldcg(q + p * plane) : 0.f;
  float v = 0.f;
#pragma unroll
  for (int p = 0; p < kRouterSplitMax; ++p)
    if (p < a.nsplit) v += u[p];
  return v + (a.bias ? __ldg(a.bias + e) : 0.f);
}

// Selection key of a logit: NaN ranks below every number (as -inf), so the
// order (key descending, id ascending) is total for any input and every CTA
// that routes the same logits derives the same selection.
__device__ __forceinline__ float route_key(float v) { return v != v ? -INFINITY : v; }

// One warp: softmax over the E logits of token t and selection of the top k
// (largest logit first, lower id first among equal logits). NV = values held
// per lane (E <= 32 * NV). Writes ids / weights to the workspace, the user
// buffers (if any) and s_ids (chunk-local copy).
template <int NV>
__device__ __forceinline__ void warp_softmax_topk(const RouteArgs& a, int t, int32_t* s_ids_row,
                                                  const float* part = nullptr) {
  const int lane = threadIdx.x & 31;
  const int E = a.E, k = a.k;
  const float* L = a.logits + (size_t)t * E;
  float v[NV];
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const int e = lane + 32 * i;
    if (e >= E)
      v[i] = -INFINITY;
    else if (part)
      v[i] = route_key(logit_from_parts(a, part, t, e));
    else if (a.nsplit > 0)
      v[i] = route_key(logit_from_planes(a, t, e));
    else
      v[i] = route_key(__ldcg(L + e));
  }
  float m = -INFINITY;
#pragma unroll
  for (int i = 0; i < NV; ++i) m = fmaxf(m, v[i]);
  m = warp_max(m);
  float ssum = 0.f;
#pragma unroll
  for (int i = 0; i < NV; ++i)
    if (lane + 32 * i < E) ssum += expf(v[i] - m);
  ssum = warp_sum(ssum);

  float my_p = 0.f, psel = 0.f;
  int my_id = 0;
  if constexpr (NV <= 4) {
    // Rank selection (E <= 128): the rank of a logit is the number of logits
    // ahead of it (larger, or equal with a lower id); the top k are ranks
    // 0..k-1. Every comparison is independent, so the warp has no serial
    // chain of k reductions.
    int rank[NV];
#pragma unroll
    for (int i = 0; i < NV; ++i) rank[i] = 0;
#pragma unroll 4
    for (int o = 0; o < 32; ++o) {
#pragma unroll
      for (int i2 = 0; i2 < NV; ++i2) {
        const float ov = __shfl_sync(0xffffffffu, v[i2], o);
        const int oe = o + 32 * i2;
#pragma unroll
        for (int i = 0; i < NV; ++i) {
          const int e = lane + 32 * i;
          rank[i] += (ov > v[i] || (ov == v[i] && oe < e)) ? 1 : 0;
        }
      }
    }
    // lane j takes the logit of rank j: walk the selected set (known to every
    // lane through ballots) and pick the holder whose rank is j
    float my_v = -INFINITY;
#pragma unroll
    for (int i2 = 0; i2 < NV; ++i2) {
      uint32_t sel = __ballot_sync(0xffffffffu, lane + 32 * i2 < E && rank[i2] < k);
      while (sel) {
        const int src = __ffs(sel) - 1;
        sel &= sel - 1;
        const int r = __shfl_sync(0xffffffffu, rank[i2], src);
        const float sv = __shfl_sync(0xffffffffu, v[i2], src);
        if (r == lane) {
          my_id = src + 32 * i2;
          my_v = sv;
        }
      }
    }
    my_p = expf(my_v - m) / ssum;
    for (int j = 0; j < k; ++j) psel += __shfl_sync(0xffffffffu, my_p, j);
  } else {
    // k rounds of a warp arg-max over the logits not yet taken
    uint32_t taken = 0;
    for (int j = 0; j < k; ++j) {
      float bv = -INFINITY;
      int bi = 0x7fffffff;
#pragma unroll
      for (int i = 0; i < NV; ++i) {
        const int e = lane + 32 * i;
        // within a lane e grows with i, so '>' keeps the lowest id of equal values
        if (e < E && !((taken >> i) & 1u) && (v[i] > bv || bi == 0x7fffffff)) {
          bv = v[i];
          bi = e;
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
        if (oi != 0x7fffffff && (bi == 0x7fffffff || ov > bv || (ov == bv && oi < bi))) {
          bv = ov;
          bi = oi;
        }
      }
      if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
      const float p = expf(bv - m) / ssum;
      if (lane == j) {
        my_p = p;
        my_id = bi;
      }
      psel += p;
    }
  }
  if (lane < k) {
    const float wv = a.renorm ? my_p / psel : my_p;
    const size_t o = (size_t)t * k + lane;
    a.ids[o] = my_id;
    a.w[o] = wv;
    if (a.ids_user) a.ids_user[o] = my_id;
    if (a.w_user) a.w_user[o] = wv;
    if (s_ids_row) s_ids_row[lane] = my_id;
  }
}

// Warp-level stable scatter of flat indices [f_begin, f_end) (ids in s_ids,
// indexed from f_begin) using per-expert running cursors.
__device__ __forceinline__ void warp_stable_scatter(const RouteArgs& a, const int32_t* s_ids, int f_begin, int f_end,
                                    int* cursor) {
  const int lane = threadIdx.x & 31;
  for (int f0 = f_begin; f0 < f_end; f0 += 32) {
    const int f = f0 + lane;
    const bool valid = f < f_end;
    const int e = valid ? s_ids[f - f_begin] : -1 - lane;
    const uint32_t peers = __match_any_sync(0xffffffffu, e);
    int pos = 0;
    if (valid) {
      pos = cursor[e] + __popc(peers & lanemask_lt());
      a.perm[pos] = f;
      a.inv_perm[f] = pos;
    }
    __syncwarp();
    if (valid && lane == __ffs(peers) - 1) cursor[e] += __popc(peers);
    __syncwarp();
  }
}

// Warp-level list of active experts (count > 0) in ascending id, plus the
// shared expert segment at the end.
__device__ __forceinline__ void warp_segments(const RouteArgs& a, const int* s_counts, const int* s_off) {
  const int lane = threadIdx.x & 31;
  int n = 0;
  for (int base = 0; base < a.E; base += 32) {
    const int e = base + lane;
    const bool act = e < a.E && s_counts[e] > 0;
    const uint32_t mask = __ballot_sync(0xffffffffu, act);
    if (act) {
      const int idx = n + __popc(mask & lanemask_lt());
      a.seg_expert[idx] = e;
      a.seg_start[idx] = s_off[e];
      a.seg_count[idx] = s_counts[e];
    }
    n += __popc(mask);
  }
  if (lane == 0) {
    if (a.has_shared) {
      a.seg_expert[n] = a.E;
      a.seg_start[n] = a.T * a.k;
      a.seg_count[n] = a.T;
      ++n;
    }
    *a.num_seg = n;
  }
}

// ------------------------------------------------------------ small path
// Single-warp finish for n = T*k <= 32 (token, rank) pairs: lane f holds pair
// f; its sorted position is the number of pairs with a lower expert id, or
// the same id and a lower flat index (a stable counting sort by rank). Also
// writes the segment list and the per-expert counts / offsets (by binary
// search over the sorted ids, all threads).
__device__ __forceinline__ void finish_tiny(const RouteArgs& a, int32_t* s_ids, int32_t* s_sorted) {
  const int tid = threadIdx.x, lane = tid & 31;
  const int n = a.T * a.k;
  if (tid < 32) {
    const int e = lane < n ? s_ids[lane] : 0x7fffffff;
    int rank = 0;
    for (int o = 0; o < n; ++o) {
      const int eo = __shfl_sync(0xffffffffu, e, o);
      rank += (eo < e || (eo == e && o < lane)) ? 1 : 0;
    }
    if (lane < n) {
      a.perm[rank] = lane;
      a.inv_perm[lane] = rank;
      s_sorted[rank] = e;
    }
    __syncwarp();
    const int se = lane < n ? s_sorted[lane] : -1;
    const bool start = lane < n && (lane == 0 || s_sorted[lane - 1] != se);
    const uint32_t mask = __ballot_sync(0xffffffffu, start);
    if (start) {
      const int idx = __popc(mask & lanemask_lt());
      const uint32_t later = mask & ~((2u << lane) - 1u);
      const int next = later ? (__ffs(later) - 1) : n;
      a.seg_expert[idx] = se;
      a.seg_start[idx] = lane;
      a.seg_count[idx] = next - lane;
    }
    if (lane == 0) {
      int ns = __popc(mask);
      if (a.has_shared) {
        a.seg_expert[ns] = a.E;
        a.seg_start[ns] = n;
        a.seg_count[ns] = a.T;
        ++ns;
      }
      *a.num_seg = ns;
    }
  }
  __syncthreads();
  // offsets[e] = number of pairs with expert < e
  for (int e = tid; e <= a.E; e += blockDim.x) {
    int lo = 0, hi = n;
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (s_sorted[mid] < e)
        lo = mid + 1;
      else
        hi = mid;
    }
    a.offsets[e] = lo;
    s_ids[32 + e] = lo;  // scratch copy for the counts
  }
  __syncthreads();
  for (int e = tid; e < a.E; e += blockDim.x) a.counts[e] = s_ids[32 + e + 1] - s_ids[32 + e];
}

// Softmax and top-k of all T tokens with every thread of the CTA (E <= 128):
// the same results, bit for bit, as warp_softmax_topk, with the work spread
// out. Each logit's rank (the number of logits of its token ahead of it:
// larger, or equal with a lower id) is counted by one thread against its
// token's row, read as broadcast 128-bit shared loads (rows padded to a
// multiple of 4 with -inf, which never ranks ahead); ranks 0..k-1 are the
// selection. The softmax maximum and denominator of a token are computed by
// one warp exactly as in warp_softmax_topk. fbuf: T*E4 + 2T + T*k floats of
// shared memory (E4 = E rounded up to a multiple of 4, block_topk_fbuf_floats).
// Writes ids / weights to a.ids, a.w, the user buffers (if any) and s_sel
// ([T][k], by rank).
__host__ __device__ inline int block_topk_fbuf_floats(int T, int E, int k) {
  return T * ((E + 3) & ~3) + 2 * T + T * k;
}
template <int NV>
__device__ __forceinline__ void block_softmax_topk(const RouteArgs& a, const float* part, float* fbuf,
                                                   int32_t* s_sel, unsigned long long* tr = nullptr) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nwarps = blockDim.x >> 5;
  const int T = a.T, E = a.E, k = a.k, E4 = (E + 3) & ~3, n4 = T * E4;
  float* lg = fbuf;       // [T][E4]
  float* mx = lg + n4;    // [T]
  float* den = mx + T;    // [T]
  float* sp = den + T;    // [T][k] probabilities by rank
  for (int i = tid; i < n4; i += blockDim.x) {
    const int t = i / E4, e = i - t * E4;
    lg[i] = e < E ? route_key(part ? logit_from_parts(a, part, t, e) : __ldcg(a.logits + (size_t)t * E + e))
                  : -INFINITY;
  }
  for (int i = tid; i < T * k; i += blockDim.x) {
    s_sel[i] = 0;  // defined even if NaN logits leave a rank unfilled
    sp[i] = 0.f;
  }
  __syncthreads();
  if (tid == 0) trace_mark(tr, 6);
  // maximum and denominator, one warp per token (as warp_softmax_topk)
  for (int t = warp; t < T; t += nwarps) {
    float v[NV];
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      const int e = lane + 32 * i;
      v[i] = (e < E) ? lg[t * E4 + e] : -INFINITY;
    }
    float m = -INFINITY;
#pragma unroll
    for (int i = 0; i < NV; ++i) m = fmaxf(m, v[i]);
    m = warp_max(m);
    float ssum = 0.f;
#pragma unroll
    for (int i = 0; i < NV; ++i)
      if (lane + 32 * i < E) ssum += expf(v[i] - m);
    ssum = warp_sum(ssum);
    if (lane == 0) {
      mx[t] = m;
      den[t] = ssum;
    }
  }
  __syncthreads();
  if (tid == 0) trace_mark(tr, 7);
  // ranks: one thread per logit
  for (int i = tid; i < n4; i += blockDim.x) {
    const int t = i / E4, e = i - t * E4;
    if (e >= E) continue;
    const float v = lg[i];
    const float4* row = reinterpret_cast<const float4*>(lg + t * E4);
    int r = 0;
    for (int q = 0; q < E4 / 4; ++q) {
      const float4 o = row[q];
      const int e0 = 4 * q;
      r += (o.x > v || (o.x == v && e0 + 0 < e)) ? 1 : 0;
      r += (o.y > v || (o.y == v && e0 + 1 < e)) ? 1 : 0;
      r += (o.z > v || (o.z == v && e0 + 2 < e)) ? 1 : 0;
      r += (o.w > v || (o.w == v && e0 + 3 < e)) ? 1 : 0;
    }
    if (r < k) {
      s_sel[t * k + r] = e;
      sp[t * k + r] = expf(v - mx[t]) / den[t];
    }
  }
  __syncthreads();
  if (tid == 0) trace_mark(tr, 8);
  // routing weights: the selected probabilities summed in rank order
  for (int o = tid; o < T * k; o += blockDim.x) {
    const int t = o / k;
    float psel = 0.f;
    for (int j = 0; j < k; ++j) psel += sp[t * k + j];
    const float p = sp[o];
    const float wv = a.renorm ? p / psel : p;
    const int id = s_sel[o];
    a.ids[o] = id;
    a.w[o] = wv;
    if (a.ids_user) a.ids_user[o] = id;
    if (a.w_user) a.w_user[o] = wv;
  }
}

// Top-k for all T tokens, the permutation and the segment list, computed by
// one CTA (all its threads). scratch: >= T*k + 3*E + 66 ints of shared
// memory, 16-byte aligned
// memory; s_scan: 33 ints of shared memory; fbuf (optional, used when
// E <= 128): T*E + 2T + T*k floats of shared memory for the block-wide
// top-k.
// TINY_ONLY: the caller guarantees T * k <= 32 (only that path is compiled).
// fbuf must be given when NV <= 4.
template <int NV>
__device__ __forceinline__ void cta_softmax_topk(const RouteArgs& a, const float* part, float* fbuf,
                                                 int32_t* s_ids, unsigned long long* tr = nullptr) {
  if constexpr (NV <= 4) {
    block_softmax_topk<NV>(a, part, fbuf, s_ids, tr);
  } else {
    const int warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
    for (int t = warp; t < a.T; t += nwarps) warp_softmax_topk<NV>(a, t, s_ids + t * a.k, part);
  }
}

template <int NV, bool TINY_ONLY = false>
__device__ __forceinline__ void route_finish_cta(const RouteArgs& a, int32_t* scratch, int* s_scan,
                                                 const float* part, unsigned long long* tr, float* fbuf) {
  const int tid = threadIdx.x, warp = tid >> 5;
  const int T = a.T, E = a.E, k = a.k;
  int32_t* s_ids = scratch;
  if (TINY_ONLY || T * k <= 32) {
    int32_t* s_sorted = s_ids + 32 + E + 1;
    cta_softmax_topk<NV>(a, part, fbuf, s_ids);
    __syncthreads();
    if (tid == 0) trace_mark(tr, 3);
    finish_tiny(a, s_ids, s_sorted);
  } else if constexpr (!TINY_ONLY) {
    // the counting sort by direct placement: the sorted position of pair f
    // is the number of pairs with a lower expert id plus those with the
    // same id and a lower flat index (stable); counts and offsets of an
    // expert likewise by counting. The pairs are read as broadcast 128-bit
    // shared loads (scratch padded to a multiple of 4 with an id past E).
    const int n = T * k, n4 = (n + 3) & ~3;
    int* s_counts = s_ids + n4;
    int* s_off = s_counts + E;
    cta_softmax_topk<NV>(a, part, fbuf, s_ids, tr);
    for (int f = n + tid; f < n4; f += blockDim.x) s_ids[f] = 0x7fffffff;
    __syncthreads();
    if (tid == 0) trace_mark(tr, 3);
    const int4* ids4 = reinterpret_cast<const int4*>(s_ids);
    for (int f = tid; f < n; f += blockDim.x) {
      const int e = s_ids[f];
      int pos = 0;
      for (int q = 0; q < n4 / 4; ++q) {
        const int4 o = ids4[q];
        const int f0 = 4 * q;
        pos += (o.x < e || (o.x == e && f0 + 0 < f)) ? 1 : 0;
        pos += (o.y < e || (o.y == e && f0 + 1 < f)) ? 1 : 0;
        pos += (o.z < e || (o.z == e && f0 + 2 < f)) ? 1 : 0;
        pos += (o.w < e || (o.w == e && f0 + 3 < f)) ? 1 : 0;
      }
      a.perm[pos] = f;
      a.inv_perm[f] = pos;
    }
    for (int e = tid; e <= E; e += blockDim.x) {
      int below = 0, at = 0;
      for (int q = 0; q < n4 / 4; ++q) {
        const int4 o = ids4[q];
        below += (o.x < e ? 1 : 0) + (o.y < e ? 1 : 0) + (o.z < e ? 1 : 0) + (o.w < e ? 1 : 0);
        at += (o.x == e ? 1 : 0) + (o.y == e ? 1 : 0) + (o.z == e ? 1 : 0) + (o.w == e ? 1 : 0);
      }
      a.offsets[e] = below;
      s_off[e] = below;
      if (e < E) {
        a.counts[e] = at;
        s_counts[e] = at;
      }
    }
    __syncthreads();
    if (warp == 0) warp_segments(a, s_counts, s_off);
    __syncthreads();
  }
}

}  // namespace moe
