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
// Two launch shapes:
//  * small T (<= kSmallRouteMaxT): one kernel; CTAs split the experts, each
//    warp computes one expert's logits for all tokens, and the last CTA to
//    finish (atomic ticket, no spinning) runs top-k, the histogram, the scan
//    and the stable scatter for the whole batch;
//  * large T: a logits kernel split over K (partial planes summed in order
//    by the next kernel), a top-k kernel per chunk of tokens that also
//    writes the chunk's expert histogram, then a scatter kernel per chunk
//    that derives its own bases from the whole histogram.
// The selection is the same rule on both; the logits' FP32 summation order
// differs between them.
#include <cfloat>
#include <cmath>

#include "route_dev.cuh"

namespace moe {

namespace {


// Router logits for T <= kSmallRouteMaxT tokens: one CTA per expert, warp p
// computes partial p of the row; the partials are summed in order (the same
// two-level sum every small-batch path uses). The last CTA to finish
// (atomic ticket, no spinning) runs top-k and the permutation for the batch.
template <int NV>
__global__ void __launch_bounds__(kLogitParts * 32) k_route_small(RouteArgs a) {
  extern __shared__ __align__(16) unsigned char smem[];
  __shared__ __align__(16) float s_part[kSmallRouteMaxT * kLogitParts];
  __shared__ int s_last;
  const int tid = threadIdx.x, warp = tid >> 5;
  const int e = blockIdx.x;
  unsigned long long* tr = tid == 0 ? a.trace : nullptr;
  trace_mark(tr, 0);
  pdl_wait();
  trace_mark(tr, 1);
  {
    // partials into shared memory laid out as part[t][0][p] (E = 1 view)
    RouteArgs one = a;
    one.E = 1;
    one.wr = a.wr + (size_t)e * a.H;
    warp_logit_partial(one, 0, warp, s_part);
  }
  __syncthreads();
  trace_mark(tr, 2);
  if (tid < a.T) {
    float v = 0.f;
#pragma unroll
    for (int p = 0; p < kLogitParts; ++p) v += s_part[tid * kLogitParts + p];
    a.logits[(size_t)tid * a.E + e] = v + (a.bias ? __ldg(a.bias + e) : 0.f);
  }

  // the last CTA to finish its logits runs the rest of the routing: the
  // threads that wrote a logit fence it before the ticket (release); the
  // ticket's taker fences after it (acquire) and the block barrier orders
  // the finish's L2 reads after that
  if (tid < a.T) __threadfence();
  __syncthreads();
  if (tid == 0) {
    s_last = (atomicAdd(a.ticket, 1u) == gridDim.x - 1);
    __threadfence();
  }
  __syncthreads();
  trace_mark(tr, 4);
  if (!s_last) return;

  // dynamic shared memory: the finish scratch (route_finish_scratch_ints)
  int32_t* scratch = reinterpret_cast<int32_t*>(smem);
  route_finish_cta<NV>(a, scratch, nullptr, tr);
  trace_mark(tr, 5);
  if (tid == 0) *a.ticket = 0u;
}

// ------------------------------------------------------------ large path
// Router logits on the tensor cores, split over K. CTA (bx, by, p) computes
// the partial dot products of 64 tokens x 64 experts over K part p (32-wide
// K chunks [p * nch / P, (p + 1) * nch / P)) and writes plane p of the
// logits workspace ([P][T][E]); the top-k kernel sums the planes in order
// and adds the bias.
//
// x is FP16, so each product x * w is exact in FP32 once w is; the FP32
// router weight is split as w = hi + lo * 2^-11 with hi = fp16(w) and
// lo = fp16((w - hi) * 2^11) (together ~22 significant bits), and
// mma.sync m16n8k16 accumulates sum x * hi and sum x * lo separately in
// FP32; the plane gets acc_hi + acc_lo * 2^-11. Warp w holds tokens
// 16 w .. 16 w + 15 and all 64 experts (8 n-tiles of 8). The next K chunk
// is loaded into registers while the current one is multiplied.
constexpr int kLgTok = 64;
constexpr int kLgExp = 64;
constexpr int kLgK = 32;
constexpr int kLgThreads = 128;
constexpr int kLgStride = kLgK + 8;  // halves per staged row: 80 bytes, conflict-free fragment reads

__device__ __forceinline__ void mma_f16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                              uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__global__ void __launch_bounds__(kLgThreads) k_router_logits_split(RouteArgs a) {
  __shared__ __align__(16) __half xs[kLgTok][kLgStride];  // [token][k]
  __shared__ __align__(16) __half wh[kLgExp][kLgStride];  // [expert][k], hi part
  __shared__ __align__(16) __half wl[kLgExp][kLgStride];  // [expert][k], lo part x 2^11
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, c = lane & 3;
  const int t0 = blockIdx.x * kLgTok, e0 = blockIdx.y * kLgExp, p = blockIdx.z;
  const int T = a.T, H = a.H, E = a.E, P = a.nsplit;
  const int nch = H / kLgK;
  const int c0 = (int)((long long)p * nch / P), c1 = (int)((long long)(p + 1) * nch / P);
  // loader roles: x row lx (16 halves at kx); router row lw (16 floats at kw)
  const int lx = tid >> 1, kx = (tid & 1) * 16;
  const int lw = tid >> 1, kw = (tid & 1) * 16;
  const bool xrow = t0 + lx < T, wrow = e0 + lw < E;
  const uint4* xsrc = reinterpret_cast<const uint4*>(a.x + (size_t)(xrow ? t0 + lx : 0) * H + kx);
  const float4* wsrc = reinterpret_cast<const float4*>(a.wr + (size_t)(wrow ? e0 + lw : 0) * H + kw);
  pdl_wait();
  float ah[8][4], al[8][4];
#pragma unroll
  for (int n = 0; n < 8; ++n)
#pragma unroll
    for (int i = 0; i < 4; ++i) ah[n][i] = al[n][i] = 0.f;
  uint4 xr0 = make_uint4(0u, 0u, 0u, 0u), xr1 = xr0;
  float4 wr[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) wr[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  auto load = [&](int ch) {
    const int o = ch * kLgK;
    if (xrow) {
      xr0 = __ldg(xsrc + o / 8);
      xr1 = __ldg(xsrc + o / 8 + 1);
    }
    if (wrow) {
#pragma unroll
      for (int i = 0; i < 4; ++i) wr[i] = __ldg(wsrc + o / 4 + i);
    }
  };
  if (c0 < c1) load(c0);
  for (int ch = c0; ch < c1; ++ch) {
    {
      *reinterpret_cast<uint4*>(&xs[lx][kx]) = xr0;
      *reinterpret_cast<uint4*>(&xs[lx][kx + 8]) = xr1;
      __align__(16) __half hh[16], hl[16];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float v[4] = {wr[i].x, wr[i].y, wr[i].z, wr[i].w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const __half h = __float2half_rn(v[j]);
          hh[4 * i + j] = h;
          hl[4 * i + j] = __float2half_rn((v[j] - __half2float(h)) * 2048.f);
        }
      }
      *reinterpret_cast<uint4*>(&wh[lw][kw]) = *reinterpret_cast<const uint4*>(&hh[0]);
      *reinterpret_cast<uint4*>(&wh[lw][kw + 8]) = *reinterpret_cast<const uint4*>(&hh[8]);
      *reinterpret_cast<uint4*>(&wl[lw][kw]) = *reinterpret_cast<const uint4*>(&hl[0]);
      *reinterpret_cast<uint4*>(&wl[lw][kw + 8]) = *reinterpret_cast<const uint4*>(&hl[8]);
    }
    __syncthreads();
    if (ch + 1 < c1) load(ch + 1);
#pragma unroll
    for (int kb = 0; kb < kLgK; kb += 16) {
      const int r = 16 * warp + g;
      const uint32_t a0 = *reinterpret_cast<const uint32_t*>(&xs[r][kb + 2 * c]);
      const uint32_t a1 = *reinterpret_cast<const uint32_t*>(&xs[r + 8][kb + 2 * c]);
      const uint32_t a2 = *reinterpret_cast<const uint32_t*>(&xs[r][kb + 2 * c + 8]);
      const uint32_t a3 = *reinterpret_cast<const uint32_t*>(&xs[r + 8][kb + 2 * c + 8]);
#pragma unroll
      for (int n = 0; n < 8; ++n) {
        const int ew = 8 * n + g;
        const uint32_t bh0 = *reinterpret_cast<const uint32_t*>(&wh[ew][kb + 2 * c]);
        const uint32_t bh1 = *reinterpret_cast<const uint32_t*>(&wh[ew][kb + 2 * c + 8]);
        const uint32_t bl0 = *reinterpret_cast<const uint32_t*>(&wl[ew][kb + 2 * c]);
        const uint32_t bl1 = *reinterpret_cast<const uint32_t*>(&wl[ew][kb + 2 * c + 8]);
        mma_f16_16816(ah[n], a0, a1, a2, a3, bh0, bh1);
        mma_f16_16816(al[n], a0, a1, a2, a3, bl0, bl1);
      }
    }
    __syncthreads();
  }
  // D fragment: rows g / g + 8 (tokens), columns 2c / 2c + 1 (experts)
  float* plane = a.logits + (size_t)p * T * E;
#pragma unroll
  for (int n = 0; n < 8; ++n)
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int t = t0 + 16 * warp + g + ((i & 2) ? 8 : 0);
      const int e = e0 + 8 * n + 2 * c + (i & 1);
      if (t < T && e < E) plane[(size_t)t * E + e] = ah[n][i] + al[n][i] * (1.f / 2048.f);
    }
}

// Softmax, top-k and the expert histogram of one chunk of kRouteChunkTokens
// tokens (one warp per token).
constexpr int kTopkThreads = 512;

template <int NV>
__global__ void __launch_bounds__(kTopkThreads) k_topk_hist(RouteArgs a) {
  extern __shared__ __align__(16) unsigned char smem[];
  const int tid = threadIdx.x, warp = tid >> 5;
  constexpr int nwarps = kTopkThreads / 32;
  const int T = a.T, E = a.E, k = a.k;
  const int c = blockIdx.x;
  const int tbeg = c * kRouteChunkTokens;
  const int tend = min(T, tbeg + kRouteChunkTokens);
  int32_t* s_ids = reinterpret_cast<int32_t*>(smem);  // [chunk tokens * k]
  int* s_hist = s_ids + kRouteChunkTokens * k;        // [E]
  pdl_wait();
  for (int i = tid; i < E; i += kTopkThreads) s_hist[i] = 0;
  for (int t = tbeg + warp; t < tend; t += nwarps) warp_softmax_topk<NV>(a, t, s_ids + (t - tbeg) * k);
  __syncthreads();
  for (int f = tid; f < (tend - tbeg) * k; f += kTopkThreads) atomicAdd(&s_hist[s_ids[f]], 1);
  __syncthreads();
  for (int i = tid; i < E; i += kTopkThreads) a.chunk_hist[(size_t)c * E + i] = s_hist[i];
}

// Stable scatter of chunk c's (token, rank) pairs. Every chunk CTA reads the
// whole histogram (independent loads, all in flight together) for its
// experts' totals and the pairs of earlier chunks; expert e's pairs of chunk
// c start at offsets[e] + (pairs of e in chunks < c). CTA 0 also writes the
// counts, offsets and the segment list.
constexpr int kScatterThreads = 256;

__global__ void __launch_bounds__(kScatterThreads) k_scatter(RouteArgs a) {
  extern __shared__ __align__(16) unsigned char smem[];
  __shared__ int s_scan[33];
  const int tid = threadIdx.x, warp = tid >> 5;
  const int c = blockIdx.x, nchunks = gridDim.x;
  const int E = a.E, k = a.k;
  int* s_before = reinterpret_cast<int*>(smem);  // [E]
  int* s_tot = s_before + E;                     // [E]
  int* s_off = s_tot + E;                        // [E + 1]
  int32_t* s_ids = s_off + E + 1;                // [chunk tokens * k]
  pdl_wait();
  for (int i = tid; i < E; i += kScatterThreads) {
    s_before[i] = 0;
    s_tot[i] = 0;
  }
  const int fbeg = c * kRouteChunkTokens * k;
  const int fend = min(a.T * k, fbeg + kRouteChunkTokens * k);
  for (int f = fbeg + tid; f < fend; f += kScatterThreads) s_ids[f - fbeg] = __ldcg(a.ids + f);
  __syncthreads();
  // (expert, part) per thread: tpe threads split an expert's chunks
  const int tpe = E >= kScatterThreads ? 1 : kScatterThreads / E;
  const int per_pass = kScatterThreads / tpe;
  for (int e0 = 0; e0 < E; e0 += per_pass) {
    const int e = e0 + tid / tpe, part = tid % tpe;
    if (tid / tpe < per_pass && e < E) {
      const int cb = (int)((long long)part * nchunks / tpe), ce = (int)((long long)(part + 1) * nchunks / tpe);
      int before = 0, tot = 0;
#pragma unroll 8
      for (int cc = cb; cc < ce; ++cc) {
        const int v = __ldcg(a.chunk_hist + (size_t)cc * E + e);
        tot += v;
        before += cc < c ? v : 0;
      }
      if (tot) atomicAdd(&s_tot[e], tot);
      if (before) atomicAdd(&s_before[e], before);
    }
  }
  __syncthreads();
  for (int i = tid; i < E; i += kScatterThreads) s_off[i] = s_tot[i];
  __syncthreads();
  block_exclusive_scan(s_off, E, s_scan);
  if (tid == 0) s_off[E] = a.T * k;
  for (int i = tid; i < E; i += kScatterThreads) s_before[i] += s_off[i];  // cursors
  __syncthreads();
  if (warp == 0) warp_stable_scatter(a, s_ids, fbeg, fend, s_before);
  if (c == 0) {
    for (int i = tid; i < E; i += kScatterThreads) {
      a.counts[i] = s_tot[i];
      a.offsets[i] = s_off[i];
    }
    if (tid == 0) a.offsets[E] = a.T * k;
    if (warp == 1) warp_segments(a, s_tot, s_off);
  }
}

template <int NV>
cudaError_t launch_route_small_nv(const RouteArgs& a, cudaStream_t s, bool pdl) {
  const size_t fbytes = (size_t)route_finish_scratch_ints(a.T, a.E, a.k) * sizeof(int);
  cudaError_t e = ensure_smem(k_route_small<NV>, fbytes);
  if (e != cudaSuccess) return e;
  return launch_ex(k_route_small<NV>, dim3(a.E), dim3(kLogitParts * 32), fbytes, s, pdl, a);
}

template <int NV>
cudaError_t launch_route_large_nv(const RouteArgs& a, cudaStream_t s, bool pdl) {
  dim3 g1((a.T + kLgTok - 1) / kLgTok, (a.E + kLgExp - 1) / kLgExp, a.nsplit);
  cudaError_t e = launch_ex(k_router_logits_split, g1, dim3(kLgThreads), 0, s, pdl, a);
  if (e != cudaSuccess) return e;
  const int nchunks = (a.T + kRouteChunkTokens - 1) / kRouteChunkTokens;
  const size_t smem2 = ((size_t)kRouteChunkTokens * a.k + (size_t)a.E) * sizeof(int);
  e = ensure_smem(k_topk_hist<NV>, smem2);
  if (e != cudaSuccess) return e;
  e = launch_ex(k_topk_hist<NV>, dim3(nchunks), dim3(kTopkThreads), smem2, s, pdl, a);
  if (e != cudaSuccess) return e;
  const size_t smem3 = ((size_t)3 * a.E + 1 + (size_t)kRouteChunkTokens * a.k) * sizeof(int);
  e = ensure_smem(k_scatter, smem3);
  if (e != cudaSuccess) return e;
  return launch_ex(k_scatter, dim3(nchunks), dim3(kScatterThreads), smem3, s, pdl, a);
}

}  // namespace

cudaError_t launch_route_small(const RouteArgs& a, cudaStream_t s, bool pdl) {
  if (a.E <= 64) return launch_route_small_nv<2>(a, s, pdl);
  if (a.E <= 128) return launch_route_small_nv<4>(a, s, pdl);
  if (a.E <= 256) return launch_route_small_nv<8>(a, s, pdl);
  if (a.E <= 512) return launch_route_small_nv<16>(a, s, pdl);
  return launch_route_small_nv<32>(a, s, pdl);
}

int router_split(int T, int E, int H, int num_sms) {
  const int tiles = ((T + kLgTok - 1) / kLgTok) * ((E + kLgExp - 1) / kLgExp);
  const int nch = H / kLgK;
  int p = 1;
  while (p < kRouterSplitMax && tiles * p < 3 * num_sms && nch >= 4 * p) p *= 2;
  return p;
}

cudaError_t launch_route_large(const RouteArgs& a, cudaStream_t s, bool pdl) {
  if (a.nsplit < 1 || a.nsplit > kRouterSplitMax || a.H % kLgK) return cudaErrorInvalidValue;
  if (a.E <= 64) return launch_route_large_nv<2>(a, s, pdl);
  if (a.E <= 128) return launch_route_large_nv<4>(a, s, pdl);
  if (a.E <= 256) return launch_route_large_nv<8>(a, s, pdl);
  if (a.E <= 512) return launch_route_large_nv<16>(a, s, pdl);
  return launch_route_large_nv<32>(a, s, pdl);
}

}  // namespace moe
