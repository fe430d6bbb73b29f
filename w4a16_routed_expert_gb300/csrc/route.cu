// Routing: router logits, softmax over all experts, top-k with ties to the
// lower expert id, routing weights, and the counting-sort permutation of the
// (token, rank) pairs by expert.
//
// Horizon RunMap report, "The complete execution path", step 2 (each token is
// routed to its selected experts); moe-stream, "Terms used here" (a router
// picks 8 of 64 experts per token). The arithmetic follows the layer
// definition in include/moe_layer.h: FP32 logits from FP16 x and FP32 router
// weights, FP32 softmax, selection decided on the FP32 logits.
//
// Two launch shapes produce identical outputs:
//  * small T (<= kSmallRouteMaxT): one kernel; CTAs split the experts, each
//    warp computes one expert's logits for all tokens, and the last CTA to
//    finish (atomic ticket, no spinning) runs top-k, the histogram, the scan
//    and the stable scatter for the whole batch;
//  * large T: a tiled logits kernel, a top-k kernel per 64-token chunk that
//    also writes the chunk's expert histogram (its last CTA turns the
//    histograms into offsets and per-chunk bases), then a scatter kernel per
//    chunk.
#include <cfloat>
#include <cmath>

#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {

constexpr int kRouteThreads = 256;

// In-place exclusive prefix sum of n ints in shared memory; returns the total.
// Called by all threads of the block. scratch: 33 ints of shared memory.
__device__ int block_exclusive_scan(int* data, int n, int* scratch) {
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

// One warp: softmax over the E logits of token t and selection of the top k
// (largest logit first, lower id first among equal logits). NV = values held
// per lane (E <= 32 * NV). Writes ids / weights to the workspace, the user
// buffers (if any) and s_ids (chunk-local copy).
template <int NV>
__device__ void warp_softmax_topk(const RouteArgs& a, int t, int32_t* s_ids_row) {
  const int lane = threadIdx.x & 31;
  const int E = a.E, k = a.k;
  const float* L = a.logits + (size_t)t * E;
  float v[NV];
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const int e = lane + 32 * i;
    v[i] = (e < E) ? __ldcg(L + e) : -INFINITY;
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

  uint32_t taken = 0;
  float my_p = 0.f, psel = 0.f;
  int my_id = 0;
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
__device__ void warp_stable_scatter(const RouteArgs& a, const int32_t* s_ids, int f_begin, int f_end,
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
__device__ void warp_segments(const RouteArgs& a, const int* s_counts, const int* s_off) {
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
__device__ void finish_tiny(const RouteArgs& a, int32_t* s_ids, int32_t* s_sorted, int* s_nseg) {
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
      *s_nseg = ns;
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

// Router logits for T <= kSmallRouteMaxT tokens: each CTA (4 warps) owns EPC
// experts; a warp covers 1/(4/EPC) of an expert row, FP32 FMA from the FP32
// router row and FP16 tokens, lane partials reduced by shuffles and shared
// memory. The last CTA to finish (atomic ticket, no spinning) runs top-k and
// the permutation for the whole batch.
template <int NV, int EPC>
__global__ void __launch_bounds__(128) k_route_small(RouteArgs a) {
  extern __shared__ __align__(16) unsigned char smem[];
  __shared__ float s_part[4][kSmallRouteMaxT];
  __shared__ int s_scan[33];
  __shared__ int s_last;
  __shared__ int s_nseg;
  constexpr int WPE = 4 / EPC;  // warps per expert
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int T = a.T, H = a.H, E = a.E, k = a.k;
  pdl_wait();

  const int e = blockIdx.x * EPC + warp / WPE;
  const int part = warp % WPE;
  float acc[kSmallRouteMaxT];
#pragma unroll
  for (int t = 0; t < kSmallRouteMaxT; ++t) acc[t] = 0.f;
  if (e < E) {
    const int span = H / WPE;  // multiple of 4 * 32 / 4 ... H % 128 == 0
    const float4* wr4 = reinterpret_cast<const float4*>(a.wr + (size_t)e * H + part * span);
    const uint2* x2 = reinterpret_cast<const uint2*>(a.x + part * span);
#pragma unroll 4
    for (int h4 = lane; h4 < span / 4; h4 += 32) {
      const float4 wv = __ldg(wr4 + h4);
#pragma unroll
      for (int t = 0; t < kSmallRouteMaxT; ++t) {
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
  }
#pragma unroll
  for (int t = 0; t < kSmallRouteMaxT; ++t)
    if (t < T) {
      const float v = warp_sum(acc[t]);
      if (lane == 0) s_part[warp][t] = v;
    }
  __syncthreads();
  if (tid < EPC * T) {
    const int ee = tid / T, t = tid % T;
    const int eg = blockIdx.x * EPC + ee;
    if (eg < E) {
      float v = 0.f;
#pragma unroll
      for (int p = 0; p < WPE; ++p) v += s_part[ee * WPE + p][t];
      a.logits[(size_t)t * E + eg] = v + (a.bias ? __ldg(a.bias + eg) : 0.f);
    }
  }

  // the last CTA to finish its logits runs the rest of the routing
  __threadfence();
  __syncthreads();
  if (tid == 0) s_last = (atomicAdd(a.ticket, 1u) == gridDim.x - 1);
  __syncthreads();
  if (!s_last) return;
  __threadfence();

  int32_t* s_ids = reinterpret_cast<int32_t*>(smem);  // [T*k] (+ scratch)
  if (T * k <= 32) {
    int32_t* s_sorted = s_ids + 32 + E + 1;
    if (warp == 0)
      for (int t = 0; t < T; ++t) warp_softmax_topk<NV>(a, t, s_ids + t * k);
    __syncthreads();
    finish_tiny(a, s_ids, s_sorted, &s_nseg);
  } else {
    int* s_counts = s_ids + T * k;
    int* s_off = s_counts + E;
    int* s_cur = s_off + E + 1;
    for (int t = warp; t < T; t += 4) warp_softmax_topk<NV>(a, t, s_ids + t * k);
    for (int i = tid; i < E; i += 128) s_counts[i] = 0;
    __syncthreads();
    for (int f = tid; f < T * k; f += 128) atomicAdd(&s_counts[s_ids[f]], 1);
    __syncthreads();
    for (int i = tid; i < E; i += 128) {
      s_off[i] = s_counts[i];
      a.counts[i] = s_counts[i];
    }
    __syncthreads();
    block_exclusive_scan(s_off, E, s_scan);
    for (int i = tid; i < E; i += 128) {
      s_cur[i] = s_off[i];
      a.offsets[i] = s_off[i];
    }
    if (tid == 0) {
      s_off[E] = T * k;
      a.offsets[E] = T * k;
    }
    __syncthreads();
    if (warp == 0) warp_stable_scatter(a, s_ids, 0, T * k, s_cur);
    if (warp == 1) warp_segments(a, s_counts, s_off);
  }
  if (tid == 0) *a.ticket = 0u;
}

// ------------------------------------------------------------ large path
// Logits tile: 32 tokens x 64 experts, K step 32; each thread 2 x 4 outputs.
__global__ void __launch_bounds__(kRouteThreads) k_router_logits_tiled(RouteArgs a) {
  __shared__ float xs[32][33];
  __shared__ float ws[32][65];
  const int tid = threadIdx.x;
  const int t0 = blockIdx.x * 32, e0 = blockIdx.y * 64;
  const int ty = tid >> 4, tx = tid & 15;
  const int T = a.T, H = a.H, E = a.E;
  pdl_wait();
  float acc[2][4];
#pragma unroll
  for (int i = 0; i < 2; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;

  for (int k0 = 0; k0 < H; k0 += 32) {
    {  // x tile: 32 tokens x 32 k, 4 halves per thread
      const int tt = tid >> 3, kk = (tid & 7) * 4;
      const int t = t0 + tt;
      float4 xv = make_float4(0.f, 0.f, 0.f, 0.f);
      if (t < T) {
        const uint2 raw = __ldg(reinterpret_cast<const uint2*>(a.x + (size_t)t * H + k0 + kk));
        const float2 lo = __half22float2(*reinterpret_cast<const __half2*>(&raw.x));
        const float2 hi = __half22float2(*reinterpret_cast<const __half2*>(&raw.y));
        xv = make_float4(lo.x, lo.y, hi.x, hi.y);
      }
      xs[kk + 0][tt] = xv.x;
      xs[kk + 1][tt] = xv.y;
      xs[kk + 2][tt] = xv.z;
      xs[kk + 3][tt] = xv.w;
    }
    {  // router tile: 64 experts x 32 k, 8 floats per thread
      const int ee = tid >> 2, kk = (tid & 3) * 8;
      const int e = e0 + ee;
      float4 w0 = make_float4(0.f, 0.f, 0.f, 0.f), w1 = w0;
      if (e < E) {
        const float4* src = reinterpret_cast<const float4*>(a.wr + (size_t)e * H + k0 + kk);
        w0 = __ldg(src);
        w1 = __ldg(src + 1);
      }
      ws[kk + 0][ee] = w0.x;
      ws[kk + 1][ee] = w0.y;
      ws[kk + 2][ee] = w0.z;
      ws[kk + 3][ee] = w0.w;
      ws[kk + 4][ee] = w1.x;
      ws[kk + 5][ee] = w1.y;
      ws[kk + 6][ee] = w1.z;
      ws[kk + 7][ee] = w1.w;
    }
    __syncthreads();
#pragma unroll 8
    for (int kk = 0; kk < 32; ++kk) {
      const float x0 = xs[kk][ty * 2 + 0], x1 = xs[kk][ty * 2 + 1];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float wv = ws[kk][tx * 4 + j];
        acc[0][j] = fmaf(x0, wv, acc[0][j]);
        acc[1][j] = fmaf(x1, wv, acc[1][j]);
      }
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int t = t0 + ty * 2 + i;
    if (t >= T) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int e = e0 + tx * 4 + j;
      if (e < E) a.logits[(size_t)t * E + e] = acc[i][j] + (a.bias ? __ldg(a.bias + e) : 0.f);
    }
  }
}

template <int NV>
__global__ void __launch_bounds__(kRouteThreads) k_topk_hist(RouteArgs a) {
  extern __shared__ __align__(16) unsigned char smem[];
  __shared__ int s_scan[33];
  __shared__ int s_last;
  const int tid = threadIdx.x, warp = tid >> 5;
  const int T = a.T, E = a.E, k = a.k;
  const int c = blockIdx.x;
  const int tbeg = c * kRouteChunkTokens;
  const int tend = min(T, tbeg + kRouteChunkTokens);
  int32_t* s_ids = reinterpret_cast<int32_t*>(smem);           // [64*k]
  int* s_hist = s_ids + kRouteChunkTokens * k;                  // [E]
  int* s_off = s_hist + E;                                       // [E+1] (last CTA)

  pdl_wait();
  for (int i = tid; i < E; i += kRouteThreads) s_hist[i] = 0;
  for (int t = tbeg + warp; t < tend; t += kRouteThreads / 32)
    warp_softmax_topk<NV>(a, t, s_ids + (t - tbeg) * k);
  __syncthreads();
  for (int f = tid; f < (tend - tbeg) * k; f += kRouteThreads) atomicAdd(&s_hist[s_ids[f]], 1);
  __syncthreads();
  for (int i = tid; i < E; i += kRouteThreads) a.chunk_hist[(size_t)c * E + i] = s_hist[i];

  __threadfence();
  __syncthreads();
  if (tid == 0) s_last = (atomicAdd(a.ticket, 1u) == gridDim.x - 1);
  __syncthreads();
  if (!s_last) return;
  __threadfence();

  const int nchunks = gridDim.x;
  // per-expert totals and per-chunk exclusive bases (relative to the expert)
  for (int e = tid; e < E; e += kRouteThreads) {
    int run = 0;
    for (int cc = 0; cc < nchunks; ++cc) {
      const int h = __ldcg(a.chunk_hist + (size_t)cc * E + e);
      a.chunk_base[(size_t)cc * E + e] = run;
      run += h;
    }
    s_hist[e] = run;
    s_off[e] = run;
    a.counts[e] = run;
  }
  __syncthreads();
  block_exclusive_scan(s_off, E, s_scan);
  if (tid == 0) {
    s_off[E] = T * k;
    a.offsets[E] = T * k;
  }
  for (int e = tid; e < E; e += kRouteThreads) a.offsets[e] = s_off[e];
  __syncthreads();
  for (int i = tid; i < nchunks * E; i += kRouteThreads) a.chunk_base[i] += s_off[i % E];
  if (warp == 0) warp_segments(a, s_hist, s_off);
  if (tid == 0) *a.ticket = 0u;
}

__global__ void __launch_bounds__(32) k_scatter(RouteArgs a) {
  extern __shared__ __align__(16) unsigned char smem[];
  const int lane = threadIdx.x;
  const int c = blockIdx.x;
  const int E = a.E, k = a.k;
  int* cur = reinterpret_cast<int*>(smem);                           // [E]
  int32_t* s_ids = cur + E;                                          // [64*k]
  pdl_wait();
  for (int e = lane; e < E; e += 32) cur[e] = a.chunk_base[(size_t)c * E + e];
  const int fbeg = c * kRouteChunkTokens * k;
  const int fend = min(a.T * k, fbeg + kRouteChunkTokens * k);
  for (int f = fbeg + lane; f < fend; f += 32) s_ids[f - fbeg] = a.ids[f];
  __syncwarp();
  warp_stable_scatter(a, s_ids, fbeg, fend, cur);
}

template <int NV>
cudaError_t launch_route_small_nv(const RouteArgs& a, cudaStream_t s, bool pdl) {
  // one expert per CTA up to 128 experts, then 2 or 4 per CTA
  const size_t fbytes = ((size_t)a.T * a.k + 3 * (size_t)a.E + 64) * sizeof(int);
  if (a.E <= 128) {
    ensure_smem(k_route_small<NV, 1>, fbytes);
    return launch_ex(k_route_small<NV, 1>, dim3(a.E), dim3(128), fbytes, s, pdl, a);
  }
  if (a.E <= 256) {
    ensure_smem(k_route_small<NV, 2>, fbytes);
    return launch_ex(k_route_small<NV, 2>, dim3((a.E + 1) / 2), dim3(128), fbytes, s, pdl, a);
  }
  ensure_smem(k_route_small<NV, 4>, fbytes);
  return launch_ex(k_route_small<NV, 4>, dim3((a.E + 3) / 4), dim3(128), fbytes, s, pdl, a);
}

template <int NV>
cudaError_t launch_route_large_nv(const RouteArgs& a, cudaStream_t s, bool pdl) {
  dim3 g1((a.T + 31) / 32, (a.E + 63) / 64);
  cudaError_t e = launch_ex(k_router_logits_tiled, g1, dim3(kRouteThreads), 0, s, pdl, a);
  if (e != cudaSuccess) return e;
  const int nchunks = (a.T + kRouteChunkTokens - 1) / kRouteChunkTokens;
  const size_t smem2 = ((size_t)kRouteChunkTokens * a.k + 2 * (size_t)a.E + 1) * sizeof(int);
  e = ensure_smem(k_topk_hist<NV>, smem2);
  if (e != cudaSuccess) return e;
  e = launch_ex(k_topk_hist<NV>, dim3(nchunks), dim3(kRouteThreads), smem2, s, pdl, a);
  if (e != cudaSuccess) return e;
  const size_t smem3 = ((size_t)a.E + (size_t)kRouteChunkTokens * a.k) * sizeof(int);
  e = ensure_smem(k_scatter, smem3);
  if (e != cudaSuccess) return e;
  return launch_ex(k_scatter, dim3(nchunks), dim3(32), smem3, s, pdl, a);
}

}  // namespace

cudaError_t launch_route_small(const RouteArgs& a, cudaStream_t s, bool pdl) {
  if (a.E <= 64) return launch_route_small_nv<2>(a, s, pdl);
  if (a.E <= 128) return launch_route_small_nv<4>(a, s, pdl);
  if (a.E <= 256) return launch_route_small_nv<8>(a, s, pdl);
  if (a.E <= 512) return launch_route_small_nv<16>(a, s, pdl);
  return launch_route_small_nv<32>(a, s, pdl);
}

cudaError_t launch_route_large(const RouteArgs& a, cudaStream_t s, bool pdl) {
  if (a.E <= 64) return launch_route_large_nv<2>(a, s, pdl);
  if (a.E <= 128) return launch_route_large_nv<4>(a, s, pdl);
  if (a.E <= 256) return launch_route_large_nv<8>(a, s, pdl);
  if (a.E <= 512) return launch_route_large_nv<16>(a, s, pdl);
  return launch_route_large_nv<32>(a, s, pdl);
}

}  // namespace moe
