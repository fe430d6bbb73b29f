// Device-side pieces of the grouped W4A16 GEMV, shared by the GEMV kernel
// (gemv.cu) and the decode megakernel (decode.cu): the producer's bulk copies
// of one work item and the consumers' register dequantisation of it.
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
#pragma once

#include "common.cuh"
#include "kernels.h"

namespace moe {

constexpr int kConsumerWarps = 8;
constexpr int kGemvThreads = (kConsumerWarps + 1) * 32;
constexpr int kMaxStages = 8;
constexpr int kHdrBytes = 256;

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

__device__ __forceinline__ uint32_t gemv_sstride(const GemvArgs& a) {
  return ((uint32_t)a.rb * a.ng * 2u + 15u) & ~15u;
}

// Producer (one thread): copy work item `item` (segment item / nrb, row block
// item % nrb) into stage `sb`, completing on `full`. A bad slot index records
// an error and completes the stage with no bytes.
template <bool DUAL>
__device__ __forceinline__ void gemv_issue_item(const GemvArgs& a, int item, int nrb, unsigned char* sb,
                                                uint64_t* full, uint64_t pol) {
  const int half_k = a.K >> 1;
  const uint32_t qbytes = (uint32_t)a.rb * half_k;
  const uint32_t sstride = gemv_sstride(a);
  const int sgi = item / nrb, rbi = item % nrb;
  const int e = a.seg_expert[sgi];
  const int slot = a.expert_to_slot[e];
  if (slot < 0 || slot >= a.num_slots) {
    record_error(a.err, MOE_DEV_ERR_BOUNDS);
    mbar_arrive_expect_tx(full, 0);
    return;
  }
  const uint8_t* rec = a.pool + (size_t)slot * a.record_bytes;
  const int r0 = rbi * a.rb;
  const int nrows = min(a.rb, a.N - r0);
  const uint32_t qb = (uint32_t)nrows * half_k;
  const uint32_t sbytes = (uint32_t)nrows * a.ng * 2u;
  mbar_arrive_expect_tx(full, DUAL ? 2u * (qb + sbytes) : qb + sbytes);
  bulk_g2s(sb, rec + a.q_off0 + (size_t)r0 * half_k, qb, full, pol);
  if (DUAL) bulk_g2s(sb + qbytes, rec + a.q_off1 + (size_t)r0 * half_k, qb, full, pol);
  unsigned char* ss = sb + (DUAL ? 2u : 1u) * qbytes;
  bulk_g2s(ss, rec + a.s_off0 + (size_t)r0 * a.ng * 2, sbytes, full, pol);
  if (DUAL) bulk_g2s(ss + sstride, rec + a.s_off1 + (size_t)r0 * a.ng * 2, sbytes, full, pol);
}

// Activations of the current token tile, pre-scaled, in registers.
template <int KCH, int NT>
struct XRegs {
  float2 xs[NT][KCH][16];
  float xsum[NT][KCH];
  int seg = -1, tb = -1;
};

// Consumer warp: all rows of item `item` this warp owns, for every token of
// the item's segment (in tiles of NT held in registers). COHERENT reads the
// activations through L2 (they may have been written by other CTAs of the
// same launch).
template <int KCH, int NT, bool DUAL, bool COHERENT>
__device__ __forceinline__ void gemv_consume_item(const GemvArgs& a, int item, int nrb, const unsigned char* sb,
                                                  XRegs<KCH, NT>& xr, int warp, int lane) {
  const int half_k = a.K >> 1;
  const uint32_t qbytes = (uint32_t)a.rb * half_k;
  const uint32_t sstride = gemv_sstride(a);
  const int lpr = a.lpr;
  const int rpw = 32 / lpr;
  const int sub = lane / lpr, cl = lane % lpr;
  const int nchunk = a.K >> 5;
  const int sgi = item / nrb, rbi = item % nrb;
  const int r0 = rbi * a.rb;
  const int nrows = min(a.rb, a.N - r0);
  const int pos0 = a.seg_start[sgi];
  const int cnt = a.seg_count[sgi];
  const uint8_t* q0 = sb;
  const uint8_t* q1 = sb + qbytes;
  const __half* sc0 = reinterpret_cast<const __half*>(sb + (DUAL ? 2u : 1u) * qbytes);
  const __half* sc1 = reinterpret_cast<const __half*>(sb + (DUAL ? 2u : 1u) * qbytes + sstride);

  for (int tb = 0; tb < cnt; tb += NT) {
    const int ntok = min(NT, cnt - tb);
    if (sgi != xr.seg || tb != xr.tb) {
#pragma unroll
      for (int i = 0; i < NT; ++i) {
        if (i < ntok) {
          const int pos = pos0 + tb + i;
          int row = pos;
          if (a.act_gather) row = (pos < a.Tk) ? (a.perm[pos] / a.k) : (pos - a.Tk);
          const __half* src = a.act + (size_t)row * a.K;
#pragma unroll
          for (int m = 0; m < KCH; ++m) {
            const int c = cl + m * lpr;
            float sum = 0.f;
            if (c < nchunk) {
              const uint4* p = reinterpret_cast<const uint4*>(src + c * 32);
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                const uint4 raw = COHERENT ? __ldcg(p + q) : __ldg(p + q);
                const __half2* hp = reinterpret_cast<const __half2*>(&raw);
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                  const float2 xv = __half22float2(hp[u]);
                  sum += xv.x + xv.y;
                  xr.xs[i][m][4 * q + u] = make_float2(xv.x * pre_scale(2 * u), xv.y * pre_scale(2 * u + 1));
                }
              }
            }
            xr.xsum[i][m] = sum;
          }
        }
      }
      xr.seg = sgi;
      xr.tb = tb;
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
                const float zp = -8.f * xr.xsum[i][m];
                acc0[i] = fmaf(s0, fmaf(dot32(w0, xr.xs[i][m]), 0x1p49f, zp), acc0[i]);
                if (DUAL) acc1[i] = fmaf(s1, fmaf(dot32(w1, xr.xs[i][m]), 0x1p49f, zp), acc1[i]);
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
              const int f = (pos < a.Tk) ? a.perm[pos] : pos;
              a.y_out[(size_t)f * a.N + r0 + rr] = acc0[i];
            }
          }
        }
      }
    }
  }
}

}  // namespace moe
