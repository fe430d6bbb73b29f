// Decode-regime grouped W4A16 GEMV over expert segments, and the weighted
// combine.
//
// Horizon RunMap report, "What is implemented": the INT4 routed experts stay
// compact in GPU memory and are executed with FP16 activations; the weights
// are expanded only in registers, never stored expanded.
//
// Work item = (expert segment, block of rb output rows). A persistent CTA
// (one per SM) walks a contiguous range of items. Its producer thread copies
// each item's INT4 rows and FP16 scales — contiguous byte ranges of the
// expert's record — into a ring of shared-memory stages with bulk async
// copies (cp.async.bulk, completion counted on an mbarrier). Eight consumer
// warps dequantise 16-byte code chunks in registers and accumulate in FP32;
// LPR lanes share a row and finish it with xor-shuffles.
//
// Dequantisation in registers. A code q in bits [4j, 4j+4) of a 32-bit word
// is isolated with one AND (nibbles 0..5) or one/two shifts (nibbles 6, 7).
// Read as an FP32 bit pattern below 2^24, the masked word is exactly
// q * 2^(p - 149), p the bit position it was left at. The activation is
// pre-scaled by 2^(100 - p) (exact), so every product is q * x * 2^-49 with
// no rounding, and the sum over a 32-code chunk is rescaled by 2^49. The zero
// point is applied once per chunk: sum_k (q_k - 8) x_k = sum_k q_k x_k -
// 8 sum_k x_k, and the chunk's FP16 scale multiplies the result (a chunk
// never straddles a scale group since 32 divides G). Products are exact and
// sums are FP32, so the only roundings are FP32 additions.
#include <algorithm>

#include "gemv_dev.cuh"

namespace moe {

namespace {

struct GemvHdr {
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  int abort_flag;
  int issued;
};

template <int KCH, int NT, bool DUAL>
__global__ void __launch_bounds__(kGemvThreads, 1) k_gemv(GemvArgs a) {
  extern __shared__ __align__(128) unsigned char smem[];
  GemvHdr* hdr = reinterpret_cast<GemvHdr*>(smem);
  unsigned char* stages = smem + kHdrBytes;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int S = a.stages;

  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&hdr->full[s], 1);
      mbar_init(&hdr->empty[s], kConsumerWarps);
    }
    hdr->abort_flag = 0;
    hdr->issued = 0;
    fence_mbar_init();
  }
  __syncthreads();
  pdl_trigger();
  pdl_wait();

  const int nseg = *a.num_seg;
  const int nrb = (a.N + a.rb - 1) / a.rb;
  const int total = nseg * nrb;
  const int ipc = (total + gridDim.x - 1) / gridDim.x;
  const int first = blockIdx.x * ipc;
  const int nitems = max(0, min(total, first + ipc) - first);

  if (warp == kConsumerWarps) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t pol = l2_policy_evict_first();
      for (int it = 0; it < nitems; ++it) {
        const int st = it % S;
        const uint32_t ph = (uint32_t)(it / S) & 1u;
        if (!mbar_wait(&hdr->empty[st], ph ^ 1u, &hdr->abort_flag, a.err)) break;
        gemv_issue_item<DUAL>(a, first + it, nrb, stages + (size_t)st * a.stage_bytes, &hdr->full[st], pol);
        hdr->issued = it + 1;
      }
    }
  } else {
    // ----------------------------------------------------------- consumers
    XRegs<KCH, NT> xr;
    for (int it = 0; it < nitems; ++it) {
      const int st = it % S;
      const uint32_t ph = (uint32_t)(it / S) & 1u;
      if (!mbar_wait(&hdr->full[st], ph, &hdr->abort_flag, a.err)) break;
      gemv_consume_item<KCH, NT, DUAL, false>(a, first + it, nrb, stages + (size_t)st * a.stage_bytes, xr, warp,
                                              lane);
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

template <int KCH, int NT, bool DUAL>
cudaError_t launch_gemv_t(const GemvArgs& a, int grid, cudaStream_t s, bool pdl) {
  const size_t smem = gemv_smem_bytes(a.stages, a.stage_bytes);
  cudaError_t e = ensure_smem(k_gemv<KCH, NT, DUAL>, smem);
  if (e != cudaSuccess) return e;
  return launch_ex(k_gemv<KCH, NT, DUAL>, dim3(grid), dim3(kGemvThreads), smem, s, pdl, a);
}

template <bool DUAL>
cudaError_t launch_gemv_d(const GemvArgs& a, int kch, int nt, int grid, cudaStream_t s, bool pdl) {
  if (kch == 1 && nt == 1) return launch_gemv_t<1, 1, DUAL>(a, grid, s, pdl);
  if (kch == 1 && nt == 2) return launch_gemv_t<1, 2, DUAL>(a, grid, s, pdl);
  if (kch == 2 && nt == 1) return launch_gemv_t<2, 1, DUAL>(a, grid, s, pdl);
  if (kch == 3 && nt == 1) return launch_gemv_t<3, 1, DUAL>(a, grid, s, pdl);
  if (kch == 4 && nt == 1) return launch_gemv_t<4, 1, DUAL>(a, grid, s, pdl);
  return cudaErrorInvalidConfiguration;
}

__global__ void __launch_bounds__(256) k_combine(CombineArgs a) {
  pdl_trigger();
  pdl_wait();
  const int t = blockIdx.y;
  const int h4 = blockIdx.x * 256 + threadIdx.x;
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
    acc.x += y.x;
    acc.y += y.y;
    acc.z += y.z;
    acc.w += y.w;
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

int gemv_lanes_per_row(int K) {
  const int chunks = K / 32;
  int lpr = 32;
  while (lpr > chunks && lpr > 4) lpr >>= 1;
  return lpr;
}

int gemv_kch(int K, int lpr) { return (K / 32 + lpr - 1) / lpr; }

size_t gemv_smem_bytes(int stages, uint32_t stage_bytes) { return kHdrBytes + (size_t)stages * stage_bytes; }

GemvPlan plan_gemv(int N, int K, int G, bool dual, int T) {
  GemvPlan p;
  p.lpr = gemv_lanes_per_row(K);
  p.kch = gemv_kch(K, p.lpr);
  const int rows_per_pass = kConsumerWarps * (32 / p.lpr);
  const int mats = dual ? 2 : 1;
  const int bytes_per_pass = mats * rows_per_pass * (K / 2);
  int m = std::max(1, 16384 / std::max(1, bytes_per_pass));
  p.rb = rows_per_pass * m;
  // keep work items multiples of 8 rows and no larger than needed
  while (p.rb > 8 && p.rb > N) p.rb >>= 1;
  p.rb = std::max(8, p.rb / 8 * 8);
  const int ng = (K + G - 1) / G;
  const uint32_t sstride = ((uint32_t)p.rb * ng * 2u + 15u) & ~15u;
  p.stage_bytes = ((uint32_t)(mats * p.rb * (K / 2)) + mats * sstride + 127u) & ~127u;
  p.stages = (int)std::min<size_t>(kMaxStages, std::max<size_t>(2, (180u * 1024u) / p.stage_bytes));
  // token tile: the pre-scaled activations of nt tokens stay in registers
  // (32 * kch * nt of them); keep that within the 288-thread register budget
  p.nt = (T > 1 && p.kch == 1) ? 2 : 1;
  return p;
}

bool gemv_plan_supported(const GemvPlan& p) {
  if (p.kch == 1) return p.nt == 1 || p.nt == 2;
  return p.kch >= 2 && p.kch <= 4 && p.nt == 1;
}

cudaError_t launch_gemv(const GemvArgs& a, bool dual, const GemvPlan& p, int grid, cudaStream_t s, bool pdl) {
  if (dual) return launch_gemv_d<true>(a, p.kch, p.nt, grid, s, pdl);
  return launch_gemv_d<false>(a, p.kch, p.nt, grid, s, pdl);
}

cudaError_t launch_combine(const CombineArgs& a, cudaStream_t s, bool pdl) {
  return launch_ex(k_combine, dim3((a.H / 4 + 255) / 256, a.T), dim3(256), 0, s, pdl, a);
}

}  // namespace moe
