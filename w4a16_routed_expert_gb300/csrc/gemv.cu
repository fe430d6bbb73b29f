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

#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {

constexpr int kConsumerWarps = 8;
constexpr int kGemvThreads = (kConsumerWarps + 1) * 32;
constexpr int kMaxStages = 8;
constexpr int kHdrBytes = 256;

struct GemvHdr {
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  int abort_flag;
  int issued;
};

// Pre-scale of the activation paired with nibble j of a word: 2^(100 - p_j),
// p_j the bit position the nibble is left at (0,4,8,12,16,20 in place; nibble
// 6 shifted to 4, nibble 7 shifted to 0).
__device__ __forceinline__ constexpr float pre_scale(int j) {
  return j == 0 ? 0x1p100f : j == 1 ? 0x1p96f : j == 2 ? 0x1p92f : j == 3 ? 0x1p88f
       : j == 4 ? 0x1p84f : j == 5 ? 0x1p80f : j == 6 ? 0x1p96f : 0x1p100f;
}

// sum over the 32 codes of a 16-byte chunk of q_k * x'_k (x' pre-scaled)
__device__ __forceinline__ float dot32(const uint4 w, const float2 (&x)[16]) {
  float2 a0 = make_float2(0.f, 0.f), a1 = make_float2(0.f, 0.f);
  const uint32_t words[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const uint32_t v = words[q];
    const float2 f01 = make_float2(__uint_as_float(v & 0xFu), __uint_as_float(v & 0xF0u));
    const float2 f23 = make_float2(__uint_as_float(v & 0xF00u), __uint_as_float(v & 0xF000u));
    const float2 f45 = make_float2(__uint_as_float(v & 0xF0000u), __uint_as_float(v & 0xF00000u));
    const float2 f67 = make_float2(__uint_as_float((v >> 20) & 0xF0u), __uint_as_float(v >> 28));
    a0 = ffma2(f01, x[4 * q + 0], a0);
    a1 = ffma2(f23, x[4 * q + 1], a1);
    a0 = ffma2(f45, x[4 * q + 2], a0);
    a1 = ffma2(f67, x[4 * q + 3], a1);
  }
  return (a0.x + a0.y) + (a1.x + a1.y);
}

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
  const int half_k = a.K >> 1;
  const uint32_t qbytes = (uint32_t)a.rb * half_k;
  const uint32_t sstride = ((uint32_t)a.rb * a.ng * 2u + 15u) & ~15u;

  if (warp == kConsumerWarps) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t pol = l2_policy_evict_first();
      for (int it = 0; it < nitems; ++it) {
        const int st = it % S;
        const uint32_t ph = (uint32_t)(it / S) & 1u;
        if (!mbar_wait(&hdr->empty[st], ph ^ 1u, &hdr->abort_flag, a.err)) break;
        const int item = first + it;
        const int sgi = item / nrb, rbi = item % nrb;
        const int e = a.seg_expert[sgi];
        int slot = a.expert_to_slot[e];
        unsigned char* sb = stages + (size_t)st * a.stage_bytes;
        if (slot < 0 || slot >= a.num_slots) {
          record_error(a.err, MOE_DEV_ERR_BOUNDS);
          mbar_arrive_expect_tx(&hdr->full[st], 0);
          hdr->issued = it + 1;
          continue;
        }
        const uint8_t* rec = a.pool + (size_t)slot * a.record_bytes;
        const int r0 = rbi * a.rb;
        const int nrows = min(a.rb, a.N - r0);
        const uint32_t qb = (uint32_t)nrows * half_k;
        const uint32_t sbytes = (uint32_t)nrows * a.ng * 2u;
        mbar_arrive_expect_tx(&hdr->full[st], DUAL ? 2u * (qb + sbytes) : qb + sbytes);
        bulk_g2s(sb, rec + a.q_off0 + (size_t)r0 * half_k, qb, &hdr->full[st], pol);
        if (DUAL) bulk_g2s(sb + qbytes, rec + a.q_off1 + (size_t)r0 * half_k, qb, &hdr->full[st], pol);
        unsigned char* ss = sb + (DUAL ? 2u : 1u) * qbytes;
        bulk_g2s(ss, rec + a.s_off0 + (size_t)r0 * a.ng * 2, sbytes, &hdr->full[st], pol);
        if (DUAL) bulk_g2s(ss + sstride, rec + a.s_off1 + (size_t)r0 * a.ng * 2, sbytes, &hdr->full[st], pol);
        hdr->issued = it + 1;
      }
    }
  } else {
    // ----------------------------------------------------------- consumers
    const int lpr = a.lpr;
    const int rpw = 32 / lpr;
    const int sub = lane / lpr, cl = lane % lpr;
    const int nchunk = a.K >> 5;
    float2 xs[NT][KCH][16];
    float xsum[NT][KCH];
    int cached_seg = -1, cached_tb = -1;

    for (int it = 0; it < nitems; ++it) {
      const int st = it % S;
      const uint32_t ph = (uint32_t)(it / S) & 1u;
      if (!mbar_wait(&hdr->full[st], ph, &hdr->abort_flag, a.err)) break;
      const int item = first + it;
      const int sgi = item / nrb, rbi = item % nrb;
      const int r0 = rbi * a.rb;
      const int nrows = min(a.rb, a.N - r0);
      const int pos0 = a.seg_start[sgi];
      const int cnt = a.seg_count[sgi];
      const unsigned char* sb = stages + (size_t)st * a.stage_bytes;
      const uint8_t* q0 = sb;
      const uint8_t* q1 = sb + qbytes;
      const __half* sc0 = reinterpret_cast<const __half*>(sb + (DUAL ? 2u : 1u) * qbytes);
      const __half* sc1 = reinterpret_cast<const __half*>(sb + (DUAL ? 2u : 1u) * qbytes + sstride);

      for (int tb = 0; tb < cnt; tb += NT) {
        const int ntok = min(NT, cnt - tb);
        if (sgi != cached_seg || tb != cached_tb) {
          // load the pre-scaled activations of this token tile into registers
#pragma unroll
          for (int i = 0; i < NT; ++i) {
            if (i < ntok) {
              const int pos = pos0 + tb + i;
              int row = pos;
              if (a.act_gather) row = (pos < a.Tk) ? (__ldg(a.perm + pos) / a.k) : (pos - a.Tk);
              const __half* src = a.act + (size_t)row * a.K;
#pragma unroll
              for (int m = 0; m < KCH; ++m) {
                const int c = cl + m * lpr;
                float sum = 0.f;
                if (c < nchunk) {
                  const uint4* p = reinterpret_cast<const uint4*>(src + c * 32);
#pragma unroll
                  for (int q = 0; q < 4; ++q) {
                    const uint4 raw = __ldg(p + q);
                    const __half2* hp = reinterpret_cast<const __half2*>(&raw);
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                      const float2 xv = __half22float2(hp[u]);
                      sum += xv.x + xv.y;
                      xs[i][m][4 * q + u] = make_float2(xv.x * pre_scale(2 * u), xv.y * pre_scale(2 * u + 1));
                    }
                  }
                }
                xsum[i][m] = sum;
              }
            }
          }
          cached_seg = sgi;
          cached_tb = tb;
        }

        for (int rbase = warp * rpw; rbase < nrows; rbase += kConsumerWarps * rpw) {
          const int rr = rbase + sub;
          const bool valid = rr < nrows;
          float acc0[NT], acc1[NT];
#pragma unroll
          for (int i = 0; i < NT; ++i) {
            acc0[i] = 0.f;
            acc1[i] = 0.f;
          }
          if (valid) {
#pragma unroll
            for (int m = 0; m < KCH; ++m) {
              const int c = cl + m * lpr;
              if (c < nchunk) {
                const int gidx = (c << 5) / a.G;
                const uint4 w0 = *reinterpret_cast<const uint4*>(q0 + (size_t)rr * half_k + c * 16);
                const float s0 = __half2float(sc0[rr * a.ng + gidx]);
                uint4 w1 = make_uint4(0, 0, 0, 0);
                float s1 = 0.f;
                if (DUAL) {
                  w1 = *reinterpret_cast<const uint4*>(q1 + (size_t)rr * half_k + c * 16);
                  s1 = __half2float(sc1[rr * a.ng + gidx]);
                }
#pragma unroll
                for (int i = 0; i < NT; ++i) {
                  if (i < ntok) {
                    const float zp = -8.f * xsum[i][m];
                    acc0[i] = fmaf(s0, fmaf(dot32(w0, xs[i][m]), 0x1p49f, zp), acc0[i]);
                    if (DUAL) acc1[i] = fmaf(s1, fmaf(dot32(w1, xs[i][m]), 0x1p49f, zp), acc1[i]);
                  }
                }
              }
            }
          }
#pragma unroll
          for (int i = 0; i < NT; ++i) {
            for (int o = lpr >> 1; o > 0; o >>= 1) {
              acc0[i] += __shfl_xor_sync(0xffffffffu, acc0[i], o);
              if (DUAL) acc1[i] += __shfl_xor_sync(0xffffffffu, acc1[i], o);
            }
          }
          if (valid) {
#pragma unroll
            for (int i = 0; i < NT; ++i) {
              if (i < ntok && cl == i) {
                const int pos = pos0 + tb + i;
                if (DUAL) {
                  const float h = silu_f(acc0[i]) * acc1[i];
                  a.h_out[(size_t)pos * a.N + r0 + rr] = __float2half_rn(h);
                } else {
                  const int f = (pos < a.Tk) ? __ldg(a.perm + pos) : pos;
                  a.y_out[(size_t)f * a.N + r0 + rr] = acc0[i];
                }
              }
            }
          }
        }
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
  if (kch == 1 && nt == 4) return launch_gemv_t<1, 4, DUAL>(a, grid, s, pdl);
  if (kch == 2 && nt == 1) return launch_gemv_t<2, 1, DUAL>(a, grid, s, pdl);
  if (kch == 2 && nt == 2) return launch_gemv_t<2, 2, DUAL>(a, grid, s, pdl);
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
  if (T <= 1)
    p.nt = 1;
  else if (p.kch == 1)
    p.nt = 4;
  else if (p.kch == 2)
    p.nt = 2;
  else
    p.nt = 1;
  return p;
}

bool gemv_plan_supported(const GemvPlan& p) {
  if (p.kch == 1) return p.nt == 1 || p.nt == 4;
  if (p.kch == 2) return p.nt == 1 || p.nt == 2;
  return (p.kch == 3 || p.kch == 4) && p.nt == 1;
}

cudaError_t launch_gemv(const GemvArgs& a, bool dual, const GemvPlan& p, int grid, cudaStream_t s, bool pdl) {
  if (dual) return launch_gemv_d<true>(a, p.kch, p.nt, grid, s, pdl);
  return launch_gemv_d<false>(a, p.kch, p.nt, grid, s, pdl);
}

cudaError_t launch_combine(const CombineArgs& a, cudaStream_t s, bool pdl) {
  return launch_ex(k_combine, dim3((a.H / 4 + 255) / 256, a.T), dim3(256), 0, s, pdl, a);
}

}  // namespace moe
