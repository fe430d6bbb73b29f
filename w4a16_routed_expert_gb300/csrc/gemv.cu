// Decode-regime grouped W4A16 GEMV over expert segments (multi-kernel path:
// one launch for gate/up + SwiGLU, one for down), and the weighted combine.
//
// Horizon RunMap report, "What is implemented": the INT4 routed experts stay
// compact in GPU memory and are executed with FP16 activations; the weights
// are expanded only in registers, never stored expanded.
//
// Work item = (expert segment, block of rb output rows). A persistent CTA
// (one per SM) walks a balanced contiguous range of items. Its producer
// thread copies each item's codes (TMA, 128-byte swizzled boxes) and FP16
// scales (bulk copy) into a ring of shared-memory stages; sixteen consumer
// warps compute the item on the tensor cores and a finisher warp writes the
// outputs from their partial sums with the device functions of
// tcgemv_dev.cuh, which the single-launch decode kernel shares, so both paths
// produce the same bits for the same plan.
#include <algorithm>

#include "tcgemv_dev.cuh"

namespace moe {

namespace {

constexpr int kGemvWarps = kTcWarps + 2;  // consumers, producer, finisher

struct GemvHdr {
  uint64_t full[kDecodeMaxStages];
  uint64_t empty[kDecodeMaxStages];
  TcRedBars red;
  int abort_flag;
  int issued;
};
static_assert(sizeof(GemvHdr) <= kHdrBytes, "GEMV header exceeds its reserved bytes");

struct GemvSmem {
  uint32_t ring, bs, cs, xs, red, total;
};
GemvSmem __host__ __device__ inline gemv_smem_layout(const TcGemvLaunch& p) {
  GemvSmem L;
  const uint32_t ns = (uint32_t)p.ns;
  const uint32_t csb = ((uint32_t)p.cs_groups * ns * 4u + 15u) & ~15u;
  L.ring = kHdrBytes;  // rounded up to 1024 in the kernel (slack below)
  L.bs = L.ring + 1024u + (uint32_t)p.stages * p.slot_bytes;
  L.cs = L.bs + (uint32_t)p.bs_chunks * ns * 64u;
  L.xs = L.cs + csb;  // group activation sums (zero points)
  L.red = L.xs + (p.a.zp ? csb : 0u);
  L.total = L.red + ((2u * (uint32_t)tc_red_words((int)ns) * 4u + 15u) & ~15u);
  return L;
}

template <bool DUAL>
__global__ void __launch_bounds__(kGemvWarps * 32, 1) k_tcgemv(const __grid_constant__ TcGemvLaunch p) {
  extern __shared__ __align__(128) unsigned char smem[];
  GemvHdr* hdr = reinterpret_cast<GemvHdr*>(smem);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int S = p.stages, NS = p.ns;
  const GemvSmem lay = gemv_smem_layout(p);
  const uint32_t sbase = smem_u32(smem);
  unsigned char* ring = smem + (((sbase + lay.ring + 1023u) & ~1023u) - sbase);
  uint4* Bs = reinterpret_cast<uint4*>(smem + lay.bs);
  float* Cs = reinterpret_cast<float*>(smem + lay.cs);
  float* Xs = p.a.zp ? reinterpret_cast<float*>(smem + lay.xs) : nullptr;
  float* red = reinterpret_cast<float*>(smem + lay.red);

  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&hdr->full[s], 1);
      mbar_init(&hdr->empty[s], kTcWarps);
    }
    tc_red_bars_init(&hdr->red);
    hdr->abort_flag = 0;
    hdr->issued = 0;
    fence_mbar_init();
  }
  __syncthreads();
  pdl_trigger();
  pdl_wait();

  const TcGemvArgs& a = p.a;
  const int nseg = *p.num_seg;
  const int nrb = (a.N + a.rb - 1) / a.rb;
  const int total = nseg * nrb;
  const int first = (int)((long long)blockIdx.x * total / gridDim.x);
  const int nitems = (int)((long long)(blockIdx.x + 1) * total / gridDim.x) - first;

  if (warp == kTcWarps) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t pol = l2_policy_evict_first();
      for (int it = 0; it < nitems; ++it) {
        const int st = it % S;
        const uint32_t ph = (uint32_t)(it / S) & 1u;
        if (!mbar_wait(&hdr->empty[st], ph ^ 1u, &hdr->abort_flag, a.err)) break;
        tc_issue_item<DUAL>(a, &p.m0, &p.m1, first + it, nrb, ring + (size_t)st * p.slot_bytes, &hdr->full[st],
                            pol);
        hdr->issued = it + 1;
      }
    }
  } else if (warp == kTcWarps + 1) {
    // ----------------------------------------------------------- finisher
    // token tile by token tile: K-part partials -> h (SwiGLU) or y
    int ti = 0;
    bool ok = true;
    for (int it = 0; it < nitems && ok; ++it) {
      const int item = first + it;
      const int sgi = item / nrb, rbi = item - sgi * nrb;
      const int cnt = a.seg_count[sgi];
      for (int tb = 0; tb < cnt; tb += kTcMaxTok) {
        const int b = ti & 1;
        int w = 1;
        if (lane == 0) w = mbar_wait(&hdr->red.full[b], (uint32_t)(ti >> 1) & 1u, &hdr->abort_flag, a.err);
        w = __shfl_sync(0xffffffffu, w, 0);
        if (!w) {
          ok = false;
          break;
        }
        tc_finish_warp<DUAL>(a, sgi, rbi, tb, min(kTcMaxTok, cnt - tb), NS, red + b * tc_red_words(NS), lane);
        __syncwarp();
        if (lane == 0) mbar_arrive(&hdr->red.free_[b]);
        ++ti;
      }
    }
  } else {
    // ----------------------------------------------------------- consumers
    // The named-barrier sequence depends only on the segment list, so every
    // consumer warp runs it in full, also after a failed (bounded) wait.
    // Barriers are only needed when the B fragments are rebuilt; partials go
    // to the finisher through the two buffers.
    int b_seg = -1, b_tb = -1;
    int ti = 0;
    for (int it = 0; it < nitems; ++it) {
      const int st = it % S;
      const uint32_t ph = (uint32_t)(it / S) & 1u;
      mbar_wait(&hdr->full[st], ph, &hdr->abort_flag, a.err);
      const unsigned char* slot = ring + (size_t)st * p.slot_bytes;
      const int item = first + it;
      const int sgi = item / nrb;
      const int cnt = a.seg_count[sgi];
      for (int tb = 0; tb < cnt; tb += kTcMaxTok) {
        const int ntok = min(kTcMaxTok, cnt - tb);
        if (sgi != b_seg || tb != b_tb) {
          tc_bar();  // every consumer warp is done with the previous B fragments
          tc_build_b<false>(a, sgi, tb, ntok, NS, Bs, Cs, tid, Xs);
          b_seg = sgi;
          b_tb = tb;
          tc_bar();
        }
        const int b = ti & 1;
        // the finisher has read this buffer (token tile ti - 2)
        if (lane == 0) mbar_wait(&hdr->red.free_[b], ((uint32_t)(ti >> 1) & 1u) ^ 1u, &hdr->abort_flag, a.err);
        __syncwarp();
        tc_compute<DUAL>(a, slot, Bs, Cs, ntok, NS, red + b * tc_red_words(NS), warp, lane, Xs);
        __syncwarp();
        if (lane == 0) mbar_arrive(&hdr->red.full[b]);
        ++ti;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&hdr->empty[st]);
    }
  }

  __syncthreads();
  if (tid == 0 && hdr->abort_flag) {
    // a wait gave up: let the copies already issued land before the CTA exits
    const int issued = hdr->issued;
    for (int s = 0; s < S && s < issued; ++s) {
      const int n = (issued - 1 - s) / S;
      mbar_wait(&hdr->full[s], (uint32_t)n & 1u, nullptr, nullptr);
    }
  }
}

__global__ void __launch_bounds__(256) k_combine(CombineArgs a) {
  pdl_trigger();
  pdl_wait();
  const int t = blockIdx.y;
  const int h4 = blockIdx.x * 256 + threadIdx.x;
  // gated shared expert: weight sigmoid(x_t . gate), the dot product summed
  // by every block of the token in the same fixed order (threads strided
  // over H, then the block's tree)
  float gw = 1.f;
  if (a.has_shared && a.gate) {
    __shared__ float part[256];
    float d = 0.f;
    for (int h = threadIdx.x; h < a.H; h += 256)
      d = fmaf(__half2float(a.xin[(size_t)t * a.H + h]), __ldg(a.gate + h), d);
    part[threadIdx.x] = d;
    __syncthreads();
    for (int o = 128; o > 0; o >>= 1) {
      if (threadIdx.x < o) part[threadIdx.x] += part[threadIdx.x + o];
      __syncthreads();
    }
    gw = 1.f / (1.f + expf(-part[0]));
  }
  if (4 * h4 >= a.H) return;
  const int Tk = a.T * a.k;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int j = 0; j < a.k; ++j) {
    const float wj = __ldg(a.w + (size_t)t * a.k + j);
    const float4 y = __ldcg(reinterpret_cast<const float4*>(a.ypart + ((size_t)t * a.k + j) * a.H) + h4);
    acc.x = fmaf(wj, y.x, acc.x);
    acc.y = fmaf(wj, y.y, acc.y);
    acc.z = fmaf(wj, y.z, acc.z);
    acc.w = fmaf(wj, y.w, acc.w);
  }
  if (a.has_shared) {
    const float4 y = __ldcg(reinterpret_cast<const float4*>(a.ypart + ((size_t)Tk + t) * a.H) + h4);
    if (a.gate) {
      acc.x = fmaf(gw, y.x, acc.x);
      acc.y = fmaf(gw, y.y, acc.y);
      acc.z = fmaf(gw, y.z, acc.z);
      acc.w = fmaf(gw, y.w, acc.w);
    } else {
      acc.x += y.x;
      acc.y += y.y;
      acc.z += y.z;
      acc.w += y.w;
    }
  }
  __half2 o01 = __floats2half2_rn(acc.x, acc.y);
  __half2 o23 = __floats2half2_rn(acc.z, acc.w);
  if (a.x) {
    const uint2 raw = __ldg(reinterpret_cast<const uint2*>(a.x + (size_t)t * a.H) + h4);
    const float2 x01 = __half22float2(*reinterpret_cast<const __half2*>(&raw.x));
    const float2 x23 = __half22float2(*reinterpret_cast<const __half2*>(&raw.y));
    const float2 v01 = __half22float2(o01), v23 = __half22float2(o23);
    o01 = __floats2half2_rn(x01.x + v01.x, x01.y + v01.y);
    o23 = __floats2half2_rn(x23.x + v23.x, x23.y + v23.y);
  }
  uint2 res;
  res.x = *reinterpret_cast<uint32_t*>(&o01);
  res.y = *reinterpret_cast<uint32_t*>(&o23);
  reinterpret_cast<uint2*>(a.out + (size_t)t * a.H)[h4] = res;
}

}  // namespace

size_t tcgemv_smem_bytes(const TcGemvLaunch& p) { return gemv_smem_layout(p).total; }

cudaError_t launch_tcgemv(const TcGemvLaunch& p, bool dual, int grid, cudaStream_t s, bool pdl) {
  const size_t smem = tcgemv_smem_bytes(p);
  if (dual) {
    cudaError_t e = ensure_smem(k_tcgemv<true>, smem);
    if (e != cudaSuccess) return e;
    return launch_ex(k_tcgemv<true>, dim3(grid), dim3(kGemvWarps * 32), smem, s, pdl, p);
  }
  cudaError_t e = ensure_smem(k_tcgemv<false>, smem);
  if (e != cudaSuccess) return e;
  return launch_ex(k_tcgemv<false>, dim3(grid), dim3(kGemvWarps * 32), smem, s, pdl, p);
}

cudaError_t launch_combine(const CombineArgs& a, cudaStream_t s, bool pdl) {
  return launch_ex(k_combine, dim3((a.H / 4 + 255) / 256, a.T), dim3(256), 0, s, pdl, a);
}

}  // namespace moe
