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

#include "route_dev.cuh"

namespace moe {

namespace {

constexpr int kRouteThreads = 256;

// Router logits for T <= kSmallRouteMaxT tokens: one CTA per expert, warp p
// computes partial p of the row; the partials are summed in order (the same
// two-level sum every small-batch path uses). The last CTA to finish
// (atomic ticket, no spinning) runs top-k and the permutation for the batch.
template <int NV>
__global__ void __launch_bounds__(kLogitParts * 32) k_route_small(RouteArgs a) {
  extern __shared__ __align__(16) unsigned char smem[];
  __shared__ __align__(16) float s_part[kSmallRouteMaxT * kLogitParts];
  __shared__ int s_scan[33];
  __shared__ int s_last;
  const int tid = threadIdx.x, warp = tid >> 5;
  const int e = blockIdx.x;
  pdl_wait();
  {
    // partials into shared memory laid out as part[t][0][p] (E = 1 view)
    RouteArgs one = a;
    one.E = 1;
    one.wr = a.wr + (size_t)e * a.H;
    warp_logit_partial(one, 0, warp, s_part);
  }
  __syncthreads();
  if (tid < a.T) {
    float v = 0.f;
#pragma unroll
    for (int p = 0; p < kLogitParts; ++p) v += s_part[tid * kLogitParts + p];
    a.logits[(size_t)tid * a.E + e] = v + (a.bias ? __ldg(a.bias + e) : 0.f);
  }

  // the last CTA to finish its logits runs the rest of the routing
  __threadfence();
  __syncthreads();
  if (tid == 0) s_last = (atomicAdd(a.ticket, 1u) == gridDim.x - 1);
  __syncthreads();
  if (!s_last) return;
  __threadfence();

  // dynamic shared memory: the finish scratch (T*k + 3E + 66 ints), then
  // the block top-k buffer (T*E + 2T + T*k floats)
  int32_t* scratch = reinterpret_cast<int32_t*>(smem);
  float* fbuf = reinterpret_cast<float*>(scratch + a.T * a.k + 3 * a.E + 66);
  route_finish_cta<NV>(a, scratch, s_scan, nullptr, nullptr, fbuf);
  if (tid == 0) *a.ticket = 0u;
}

// ------------------------------------------------------------ large path
// Logits tile: 32 tokens x 64 experts per CTA (128 threads, 4 x 4 outputs
// each), K in steps of 32 staged through shared memory; FP32 FMA.
__global__ void __launch_bounds__(128) k_router_logits_tiled(RouteArgs a) {
  __shared__ __align__(16) float xs[32][32 + 4];  // [k][token]
  __shared__ __align__(16) float ws[32][64 + 4];  // [k][expert]
  const int tid = threadIdx.x;
  const int t0 = blockIdx.x * 32, e0 = blockIdx.y * 64;
  const int ty = tid >> 4, tx = tid & 15;  // tokens 4*ty.., experts 4*tx..
  const int T = a.T, H = a.H, E = a.E;
  pdl_wait();
  float acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;

  for (int k0 = 0; k0 < H; k0 += 32) {
    {  // x tile: 32 tokens x 32 k = 1024 halves, 8 per thread
      const int tt = tid >> 2, kk = (tid & 3) * 8;
      const int t = t0 + tt;
      uint4 raw = make_uint4(0, 0, 0, 0);
      if (t < T) raw = __ldg(reinterpret_cast<const uint4*>(a.x + (size_t)t * H + k0 + kk));
      const __half2* hp = reinterpret_cast<const __half2*>(&raw);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const float2 v = __half22float2(hp[u]);
        xs[kk + 2 * u][tt] = v.x;
        xs[kk + 2 * u + 1][tt] = v.y;
      }
    }
#pragma unroll
    for (int rep = 0; rep < 4; ++rep) {  // router tile: 64 experts x 32 k, 16 floats per thread
      const int idx = rep * 128 + tid;
      const int ee = idx >> 3, kk = (idx & 7) * 4;
      const int e = e0 + ee;
      float4 w = make_float4(0.f, 0.f, 0.f, 0.f);
      if (e < E) w = __ldg(reinterpret_cast<const float4*>(a.wr + (size_t)e * H + k0 + kk));
      ws[kk + 0][ee] = w.x;
      ws[kk + 1][ee] = w.y;
      ws[kk + 2][ee] = w.z;
      ws[kk + 3][ee] = w.w;
    }
    __syncthreads();
#pragma unroll 8
    for (int kk = 0; kk < 32; ++kk) {
      const float4 xv = *reinterpret_cast<const float4*>(&xs[kk][4 * ty]);
      const float4 wv = *reinterpret_cast<const float4*>(&ws[kk][4 * tx]);
      const float xa[4] = {xv.x, xv.y, xv.z, xv.w};
      const float wa[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(xa[i], wa[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int t = t0 + 4 * ty + i;
    if (t >= T) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int e = e0 + 4 * tx + j;
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
  // per-expert totals and per-chunk exclusive bases (relative to the expert):
  // one warp per expert, lane i scans a contiguous block of chunks, then a
  // warp exclusive scan of the block totals
  {
    const int lane = tid & 31;
    const int per = (nchunks + 31) / 32;
    for (int e = warp; e < E; e += kRouteThreads / 32) {
      const int c0 = lane * per;
      int local = 0;
      for (int i = 0; i < per; ++i) {
        const int cc = c0 + i;
        if (cc < nchunks) local += __ldcg(a.chunk_hist + (size_t)cc * E + e);
      }
      int incl = local;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      int run = incl - local;
      for (int i = 0; i < per; ++i) {
        const int cc = c0 + i;
        if (cc < nchunks) {
          const int h = __ldcg(a.chunk_hist + (size_t)cc * E + e);
          a.chunk_base[(size_t)cc * E + e] = run;
          run += h;
        }
      }
      const int total = __shfl_sync(0xffffffffu, incl, 31);
      if (lane == 0) {
        s_hist[e] = total;
        s_off[e] = total;
        a.counts[e] = total;
      }
    }
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
  const size_t fbytes = ((size_t)a.T * a.k + 3 * (size_t)a.E + 66) * sizeof(int) +
                        ((size_t)a.T * a.E + 2 * (size_t)a.T + (size_t)a.T * a.k) * sizeof(float);
  cudaError_t e = ensure_smem(k_route_small<NV>, fbytes);
  if (e != cudaSuccess) return e;
  return launch_ex(k_route_small<NV>, dim3(a.E), dim3(kLogitParts * 32), fbytes, s, pdl, a);
}

template <int NV>
cudaError_t launch_route_large_nv(const RouteArgs& a, cudaStream_t s, bool pdl) {
  dim3 g1((a.T + 31) / 32, (a.E + 63) / 64);
  cudaError_t e = launch_ex(k_router_logits_tiled, g1, dim3(128), 0, s, pdl, a);
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
