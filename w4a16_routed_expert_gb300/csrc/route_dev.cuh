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

// Bitonic sort of the warp's 32 NV (key, id) pairs, best first: larger key
// first, lower id first among equal keys (ids distinct, so the order is
// total). Position NV * lane + i is register i of the lane; pairs at
// distance d < NV are exchanged within a lane, the others with lane ^ (d / NV).
// A pair of a block of `size` positions is put in order when the block's
// index bit `size` is 0, in reverse otherwise.
template <int NV>
__device__ __forceinline__ void warp_bitonic_best_first(float (&key)[NV], int (&id)[NV]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int size = 2; size <= 32 * NV; size <<= 1) {
#pragma unroll
    for (int d = size >> 1; d > 0; d >>= 1) {
      if (d < NV) {
#pragma unroll
        for (int i = 0; i < NV; ++i) {
          if (i & d) continue;
          const int j = i | d;
          const bool fwd = ((NV * lane + i) & size) == 0;
          const bool j_ahead = key[j] > key[i] || (key[j] == key[i] && id[j] < id[i]);
          if (fwd == j_ahead) {
            const float tk = key[i];
            key[i] = key[j];
            key[j] = tk;
            const int ti = id[i];
            id[i] = id[j];
            id[j] = ti;
          }
        }
      } else {
        const int ld = d / NV;
        const bool lower = (lane & ld) == 0;
        const bool fwd = ((NV * lane) & size) == 0;
#pragma unroll
        for (int i = 0; i < NV; ++i) {
          const float ok = __shfl_xor_sync(0xffffffffu, key[i], ld);
          const int oi = __shfl_xor_sync(0xffffffffu, id[i], ld);
          const bool other_ahead = ok > key[i] || (ok == key[i] && oi < id[i]);
          // the lower position of a forward pair keeps the better element
          if ((lower == fwd) == other_ahead) {
            key[i] = ok;
            id[i] = oi;
          }
        }
      }
    }
  }
}

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
    // Sort selection (E <= 128): the warp's 32 NV (logit, id) pairs sorted
    // best first by a bitonic network in registers; rank j then sits in
    // lane j / NV, register j % NV, and lane j < k takes it.
    int id[NV];
#pragma unroll
    for (int i = 0; i < NV; ++i) id[i] = lane + 32 * i;
    warp_bitonic_best_first<NV>(v, id);
    float my_v = -INFINITY;
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      const float sv = __shfl_sync(0xffffffffu, v[i], lane / NV);
      const int si = __shfl_sync(0xffffffffu, id[i], lane / NV);
      if (lane % NV == i) {
        my_v = sv;
        my_id = si;
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

// Top-k for all T tokens, the permutation and the segment list, computed by
// one CTA (all its threads), one warp per token for the top-k.
// scratch: route_finish_scratch_ints(T, E, k) ints of shared memory.
// TINY_ONLY: the caller guarantees T * k <= 32 (only that path is compiled).
template <int NV>
__device__ __forceinline__ void cta_softmax_topk(const RouteArgs& a, const float* part, int32_t* s_ids) {
  const int warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  for (int t = warp; t < a.T; t += nwarps) warp_softmax_topk<NV>(a, t, s_ids + t * a.k, part);
}

__host__ __device__ inline int route_finish_scratch_ints(int T, int E, int k) { return T * k + 3 * E + 66; }

template <int NV, bool TINY_ONLY = false>
__device__ __forceinline__ void route_finish_cta(const RouteArgs& a, int32_t* scratch, const float* part,
                                                 unsigned long long* tr) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int T = a.T, E = a.E, k = a.k;
  int32_t* s_ids = scratch;
  if (TINY_ONLY || T * k <= 32) {
    int32_t* s_sorted = s_ids + 32 + E + 1;
    cta_softmax_topk<NV>(a, part, s_ids);
    __syncthreads();
    if (tid == 0) trace_mark(tr, 3);
    finish_tiny(a, s_ids, s_sorted);
  } else if constexpr (!TINY_ONLY) {
    // the counting sort: counts by shared-memory atomic adds (integers: the
    // order of the adds does not matter), then one warp scans them into
    // offsets and places the pairs in flat order, 32 at a time (stable)
    const int n = T * k;
    int* s_counts = s_ids + n;    // [E]
    int* s_off = s_counts + E;    // [E + 1]
    int* s_cur = s_off + E + 1;   // [E] placement cursors
    for (int e = tid; e < E; e += blockDim.x) s_counts[e] = 0;
    cta_softmax_topk<NV>(a, part, s_ids);
    __syncthreads();
    if (tid == 0) trace_mark(tr, 3);
    for (int f = tid; f < n; f += blockDim.x) atomicAdd(&s_counts[s_ids[f]], 1);
    __syncthreads();
    if (warp == 0) {
      // lane l scans the experts [l * per, (l + 1) * per)
      const int per = (E + 31) / 32, e0 = lane * per;
      int sum = 0;
      for (int i = 0; i < per; ++i)
        if (e0 + i < E) sum += s_counts[e0 + i];
      int incl = sum;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      int run = incl - sum;
      for (int i = 0; i < per; ++i) {
        const int e = e0 + i;
        if (e < E) {
          const int c = s_counts[e];
          s_off[e] = run;
          s_cur[e] = run;
          a.offsets[e] = run;
          a.counts[e] = c;
          run += c;
        }
      }
      if (lane == 31) {
        s_off[E] = incl;
        a.offsets[E] = incl;
      }
      __syncwarp();
      warp_stable_scatter(a, s_ids, 0, n, s_cur);
      warp_segments(a, s_counts, s_off);
    }
    __syncthreads();
  }
}

}  // namespace moe
