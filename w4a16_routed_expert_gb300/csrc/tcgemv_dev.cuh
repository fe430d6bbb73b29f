// Tensor-core grouped GEMV for small token counts (decode regime): the INT4
// codes of a work item are dequantised in registers straight into the FP16
// A fragments of mma.sync m16n8k16, with the item's tokens (up to 8) as the
// n = 8 columns of B. FP32 accumulation.
//
// Why not FP32 FMAs: on this part an SM must retire ~46-58 codes per cycle
// to keep pace with HBM at batch 1, while a dequantise-and-FMA inner loop
// costs ~2.8 instructions per code (at most ~46 codes per cycle at a perfect
// issue rate). Here a code costs about one instruction:
//  * one 32-bit word holds codes 8c..8c+7 of a row's 32-code chunk (low
//    nibble = even k). Two LOP3s with magic constants put nibble pairs into
//    FP16 halves as (1024 + q) for even k and (64 + q) for odd k, and one
//    shift brings the upper byte down: 5 instructions per 8 codes;
//  * the k order inside a chunk is permuted identically for A and B, so each
//    LOP3 result is directly one A register: k-step 0 of chunk j takes codes
//    (8c+0, 8c+4) and (8c+1, 8c+5), k-step 1 codes (8c+2, 8c+6) and
//    (8c+3, 8c+7), for fragment column pairs (2c, 2c+1) and (2c+8, 2c+9);
//  * the offsets are removed per quantisation group: sum_k (q_k - 8) x_k =
//    D - C with D the group's MMA sum and C = 1032 * sum_{k even} x_k +
//    72 * sum_{k odd} x_k, a per-(group, token) constant of the activations;
//  * every product (1024 + q) x or (64 + q) x is exact in FP32.
// The codes arrive by TMA in 128-byte boxes with the 128-byte swizzle, so
// ldmatrix reads each 8-row x 16-byte fragment without bank conflicts.
//
// Work split inside an item of rb rows (rt = rb / 16 row tiles) and M
// matrices (2 for gate/up, 1 for down): consumer warp w takes row tile
// w / kparts and the quantisation groups of K part w % kparts (kparts =
// kTcWarps / rt), for all M matrices at once (one B fragment load serves
// both gate and up). Partial sums go to shared memory and are reduced over
// the K parts in a fixed order; the gate/up epilogue applies SwiGLU. Sixteen
// consumer warps per SM: a warp's dequantise -> MMA chain is latency bound,
// and measured throughput per SM grows with the number of such warps.
#pragma once

#include <cuda.h>

#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace moe {

constexpr int kTcWarps = 16;         // consumer warps sharing an item
constexpr int kTcMaxRowTiles = 8;    // 16-row tiles per item (kparts = kTcWarps / tiles >= 2)
constexpr int kTcThreads = kTcWarps * 32;
constexpr int kTcMaxTok = 8;         // tokens per MMA column tile
constexpr int kHdrBytes = 256;       // mbarrier header at the start of dynamic shared memory

// TMA tensor load with an L2 cache policy.
__device__ __forceinline__ void tma_load_3d_hint(void* dst, const CUtensorMap* tm, int c0, int c1, int c2,
                                                 uint64_t* bar, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(smem_u32(dst)),
      "l"(tm), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar)), "l"(pol)
      : "memory");
}

__device__ __forceinline__ void ldmatrix_x4(uint32_t (&r)[4], uint32_t saddr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(saddr));
}

__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                          uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t lop3_and_or(uint32_t a, uint32_t mask, uint32_t c) {
  uint32_t r;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(r) : "r"(a), "r"(mask), "r"(c));
  return r;
}

// The four A registers of one 32-bit code word: (1024 + q) for codes 0, 4 /
// 2, 6 and (64 + q) for codes 1, 5 / 3, 7 of the word.
struct DeqWord {
  uint32_t h04, h15, h26, h37;
};
__device__ __forceinline__ DeqWord dequant_word(uint32_t w) {
  DeqWord d;
  d.h04 = lop3_and_or(w, 0x000F000Fu, 0x64006400u);
  d.h15 = lop3_and_or(w, 0x00F000F0u, 0x54005400u);
  const uint32_t w8 = w >> 8;
  d.h26 = lop3_and_or(w8, 0x000F000Fu, 0x64006400u);
  d.h37 = lop3_and_or(w8, 0x00F000F0u, 0x54005400u);
  return d;
}

// Shared-memory layout of one ring slot (an item): M code matrices of nbox
// swizzled boxes (128 bytes x rb rows each), then M scale blocks of
// rb x ng FP16 (sstride bytes apart).
__device__ __forceinline__ uint32_t tc_code_off(const TcGemvArgs& a, int m, int row, int chunk) {
  return (uint32_t)m * a.code_mat_bytes + (uint32_t)(chunk >> 3) * (128u * (uint32_t)a.rb) + (uint32_t)row * 128u +
         ((uint32_t)((chunk & 7) ^ (row & 7)) << 4);
}

// Producer (one thread): copy work item `item` (segment item / nrb, row block
// item % nrb) of M matrices into slot `sb`, completing on `full`. A bad slot
// index records an error and completes the stage with no bytes.
template <bool DUAL>
__device__ __forceinline__ void tc_issue_item(const TcGemvArgs& a, const CUtensorMap* m0, const CUtensorMap* m1,
                                              int item, int nrb, unsigned char* sb, uint64_t* full, uint64_t pol) {
  constexpr int M = DUAL ? 2 : 1;
  const int sgi = item / nrb, rbi = item % nrb;
  const int e = a.seg_expert[sgi];
  const int slot = a.expert_to_slot[e];
  if (slot < 0 || slot >= a.num_slots) {
    record_error(a.err, MOE_DEV_ERR_BOUNDS);
    mbar_arrive_expect_tx(full, 0);
    return;
  }
  const int r0 = rbi * a.rb;
  const int nrows = min(a.rb, a.N - r0);
  const uint32_t sbytes = (uint32_t)nrows * a.ng * 2u;
  const uint32_t zbytes = a.zp ? (uint32_t)nrows * a.ng : 0u;  // a multiple of 16 (nrows is)
  mbar_arrive_expect_tx(full, M * (a.code_mat_bytes + sbytes + zbytes));
  for (int b = 0; b < a.nbox; ++b) {
    tma_load_3d_hint(sb + b * 128u * a.rb, m0, b * 128, r0, slot, full, pol);
    if (DUAL) tma_load_3d_hint(sb + a.code_mat_bytes + b * 128u * a.rb, m1, b * 128, r0, slot, full, pol);
  }
  const uint8_t* rec = a.pool + (size_t)slot * a.record_bytes;
  unsigned char* ss = sb + M * a.code_mat_bytes;
  bulk_g2s(ss, rec + a.s_off0 + (size_t)r0 * a.ng * 2, sbytes, full, pol);
  if (DUAL) bulk_g2s(ss + a.sstride, rec + a.s_off1 + (size_t)r0 * a.ng * 2, sbytes, full, pol);
  if (a.zp) {
    // zero-point rows after the scale blocks
    unsigned char* zs = ss + M * a.sstride;
    bulk_g2s(zs, rec + a.z_off0 + (size_t)r0 * a.ng, zbytes, full, pol);
    if (DUAL) bulk_g2s(zs + a.zstride, rec + a.z_off1 + (size_t)r0 * a.ng, zbytes, full, pol);
  }
}

// K-part partial sums in shared memory: per (consumer warp, matrix) a block
// of 16 rows x NS tokens, blocks tc_red_block(NS) floats apart. The odd
// stride puts the K parts of one output in distinct banks for the finish.
__host__ __device__ constexpr int tc_red_block(int ns) { return 16 * ns + 1; }
// floats of one partial buffer (two matrices)
__host__ __device__ constexpr int tc_red_words(int ns) { return kTcWarps * 2 * tc_red_block(ns); }

// Consumer-only barrier (the kTcWarps consumer warps, named barrier 1).
__device__ __forceinline__ void tc_bar() { asm volatile("bar.sync 1, %0;" ::"r"(kTcThreads) : "memory"); }

// B operand of a token tile: tokens tb .. tb + ntok - 1 of segment sgi, in
// fragment order Bs[(chunk * NS + n) * 4 + c] = the four half2 (x0, x4),
// (x1, x5), (x2, x6), (x3, x7) of codes 32 chunk + 8 c .. + 7 of token n
// (zero for n >= ntok or beyond K), and the group constants
// Cs[gi * NS + n] = 1032 sum_even x + 72 sum_odd x. All consumer threads
// call it (tc = 0 .. kTcThreads - 1; it contains one consumer barrier); the
// caller synchronises afterwards.
template <bool COHERENT>
__device__ __forceinline__ void tc_build_b(const TcGemvArgs& a, int sgi, int tb, int ntok, int NS, uint4* Bs,
                                           float* Cs, int tc, float* Xs = nullptr) {
  const int K = a.K;
  const int nchunk = K >> 5, nch_pad = (nchunk + 1) & ~1;
  const int pos0 = a.seg_start[sgi] + tb;
  const int total = nch_pad * NS * 4;
  const int lns = NS == 2 ? 1 : (NS == 4 ? 2 : 3);  // NS is 2, 4 or 8
  for (int e = tc; e < total; e += kTcThreads) {
    const int c = e & 3, n = (e >> 2) & (NS - 1), j = e >> (2 + lns);
    uint4 o = make_uint4(0u, 0u, 0u, 0u);
    if (n < ntok && j < nchunk) {
      const int pos = pos0 + n;
      int row = pos;
      if (a.act_gather) row = (pos < a.Tk) ? (a.perm[pos] / a.k) : (pos - a.Tk);
      const uint4* src = reinterpret_cast<const uint4*>(a.act + (size_t)row * K + 32 * j + 8 * c);
      const uint4 v = COHERENT ? __ldcg(src) : __ldg(src);
      // halves h0..h7 in v.x = (h0, h1), v.y = (h2, h3), v.z = (h4, h5), v.w = (h6, h7)
      o.x = __byte_perm(v.x, v.z, 0x5410);  // (h0, h4)
      o.y = __byte_perm(v.x, v.z, 0x7632);  // (h1, h5)
      o.z = __byte_perm(v.y, v.w, 0x5410);  // (h2, h6)
      o.w = __byte_perm(v.y, v.w, 0x7632);  // (h3, h7)
    }
    Bs[e] = o;
  }
  tc_bar();
  // group constants from the staged fragments, one (group, token) per
  // thread, fixed summation order: chunks, then c, then the four pairs
  const int cpg = a.G >> 5;
  for (int q = tc; q < a.ng * NS; q += kTcThreads) {
    const int gi = q >> lns, n = q & (NS - 1);
    float se = 0.f, so = 0.f;
    if (n < ntok) {
      const int j1 = min((gi + 1) * cpg, nchunk);
      for (int j = gi * cpg; j < j1; ++j)
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const uint4 o = Bs[(j * NS + n) * 4 + c];
          const float2 p0 = __half22float2(*reinterpret_cast<const __half2*>(&o.x));  // x0, x4
          const float2 p1 = __half22float2(*reinterpret_cast<const __half2*>(&o.y));  // x1, x5
          const float2 p2 = __half22float2(*reinterpret_cast<const __half2*>(&o.z));  // x2, x6
          const float2 p3 = __half22float2(*reinterpret_cast<const __half2*>(&o.w));  // x3, x7
          se += (p0.x + p0.y) + (p2.x + p2.y);
          so += (p1.x + p1.y) + (p3.x + p3.y);
        }
    }
    Cs[q] = 1032.f * se + 72.f * so;
    if (Xs) Xs[q] = se + so;  // the group's sum of activations (zero points)
  }
}

// One consumer warp's part of an item (row tile w / kparts, K part
// w % kparts) for the current token tile; partial sums to red
// ([warp][m][16 rows][NS tokens]). CPG = chunks per quantisation group
// (G / 32: 1, 2 or 4), so the group walk has a fixed trip count. A step
// loads one chunk pair (ldmatrix x4): half a group at G = 64 / 128, two
// groups at G = 32. ZP: the group's zero point z enters as
// sum_k (q - z) x_k = (D - C) + (8 - z) X, X the group's activation sum.
template <bool DUAL, int CPG, bool ZP>
__device__ __forceinline__ void tc_compute_g(const TcGemvArgs& a, const unsigned char* sb, const uint4* Bs,
                                             const float* Cs, const float* Xs, int ntok, int NS, float* red,
                                             int warp, int lane) {
  constexpr int M = DUAL ? 2 : 1;
  const int u = warp >> a.lkparts, kp = warp & (a.kparts - 1);
  const int g = lane >> 2, c = lane & 3;
  const int nchunk = a.K >> 5;
  // ldmatrix source of this lane: matrix lane / 8 = rows (mi & 1) * 8 + lane % 8 of chunk j + (mi >> 1).
  // Chunk pairs start at even j, so the pair's box is j / 8 and the
  // swizzled 16-byte column is ((j % 8) + (mi >> 1)) ^ (lane % 8).
  const int mi = lane >> 3, x7 = lane & 7, hi = mi >> 1;
  const uint32_t boxb = 128u * (uint32_t)a.rb;
  const uint32_t lbase = smem_u32(sb) + (uint32_t)(u * 16 + (mi & 1) * 8 + x7) * 128u;
  const uint32_t hx4 = (uint32_t)((hi ^ x7) << 4);  // (j % 8 + hi) ^ x7 = (j & 6) ^ (hi ^ x7) for even j
  const unsigned char* sc = sb + M * a.code_mat_bytes;
  const unsigned char* zc = sc + M * a.sstride;  // zero-point rows (ZP)
  const bool has_tok = g < ntok;
  const uint4* bsl = Bs + g * 4 + c;  // token g, column group c; chunk j at + j * NS * 4
  const int bstep = NS * 4;
  const int rg = u * 16 + g;
  float acc[M][4];
#pragma unroll
  for (int m = 0; m < M; ++m)
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[m][i] = 0.f;

  // group epilogue: remove the offsets (and the zero points), apply the scales
  auto epilogue = [&](int gi, const float (&d)[M][4]) {
    const float cc0 = (2 * c < NS) ? Cs[gi * NS + 2 * c] : 0.f;
    const float cc1 = (2 * c + 1 < NS) ? Cs[gi * NS + 2 * c + 1] : 0.f;
    float x0 = 0.f, x1 = 0.f;
    if (ZP) {
      x0 = (2 * c < NS) ? Xs[gi * NS + 2 * c] : 0.f;
      x1 = (2 * c + 1 < NS) ? Xs[gi * NS + 2 * c + 1] : 0.f;
    }
#pragma unroll
    for (int m = 0; m < M; ++m) {
      const __half* scm = reinterpret_cast<const __half*>(sc + m * a.sstride);
      const float s0 = __half2float(scm[rg * a.ng + gi]);
      const float s8 = __half2float(scm[(rg + 8) * a.ng + gi]);
      if (ZP) {
        const unsigned char* zm = zc + m * a.zstride;
        const float o0 = 8.f - (float)zm[rg * a.ng + gi], o8 = 8.f - (float)zm[(rg + 8) * a.ng + gi];
        acc[m][0] = fmaf(s0, fmaf(o0, x0, d[m][0] - cc0), acc[m][0]);
        acc[m][1] = fmaf(s0, fmaf(o0, x1, d[m][1] - cc1), acc[m][1]);
        acc[m][2] = fmaf(s8, fmaf(o8, x0, d[m][2] - cc0), acc[m][2]);
        acc[m][3] = fmaf(s8, fmaf(o8, x1, d[m][3] - cc1), acc[m][3]);
      } else {
        acc[m][0] = fmaf(s0, d[m][0] - cc0, acc[m][0]);
        acc[m][1] = fmaf(s0, d[m][1] - cc1, acc[m][1]);
        acc[m][2] = fmaf(s8, d[m][2] - cc0, acc[m][2]);
        acc[m][3] = fmaf(s8, d[m][3] - cc1, acc[m][3]);
      }
    }
  };

  if constexpr (CPG == 1) {
    // G = 32: a chunk pair is two groups; the K parts take pairs of groups
    const int npair = (a.ng + 1) >> 1;
    const int p0 = (kp * npair) >> a.lkparts, p1 = ((kp + 1) * npair) >> a.lkparts;
    for (int pp = p0; pp < p1; ++pp) {
      const int j = 2 * pp;  // chunk of group j; group j + 1 (if any) is chunk j + 1
      float d0[M][4], d1[M][4];
#pragma unroll
      for (int m = 0; m < M; ++m)
#pragma unroll
        for (int i = 0; i < 4; ++i) d0[m][i] = d1[m][i] = 0.f;
      uint4 b0 = make_uint4(0u, 0u, 0u, 0u), b1 = b0;
      if (has_tok) {
        b0 = bsl[j * bstep];
        b1 = bsl[(j + 1) * bstep];  // zero past the last chunk (the fragments are padded to a pair)
      }
      const uint32_t off = lbase + (uint32_t)(j >> 3) * boxb + ((((uint32_t)j << 4) & 0x60u) ^ hx4);
#pragma unroll
      for (int m = 0; m < M; ++m) {
        uint32_t r[4];
        ldmatrix_x4(r, off + (uint32_t)m * a.code_mat_bytes);
        const DeqWord w0 = dequant_word(r[0]), w1 = dequant_word(r[1]);
        mma_16816(d0[m], w0.h04, w1.h04, w0.h15, w1.h15, b0.x, b0.y);
        mma_16816(d0[m], w0.h26, w1.h26, w0.h37, w1.h37, b0.z, b0.w);
        const DeqWord w2 = dequant_word(r[2]), w3 = dequant_word(r[3]);
        mma_16816(d1[m], w2.h04, w3.h04, w2.h15, w3.h15, b1.x, b1.y);
        mma_16816(d1[m], w2.h26, w3.h26, w2.h37, w3.h37, b1.z, b1.w);
      }
      epilogue(j, d0);
      if (j + 1 < a.ng) epilogue(j + 1, d1);
    }
  } else {
    const int g0 = (kp * a.ng) >> a.lkparts, g1 = ((kp + 1) * a.ng) >> a.lkparts;
    // group by group: each chunk pair is loaded (ldmatrix + B fragments),
    // dequantised and multiplied; one accumulator chain per matrix and group
    for (int gi = g0; gi < g1; ++gi) {
      float d[M][4];
#pragma unroll
      for (int m = 0; m < M; ++m)
#pragma unroll
        for (int i = 0; i < 4; ++i) d[m][i] = 0.f;
      const int jg = gi * CPG;
#pragma unroll
      for (int pp = 0; pp < CPG / 2; ++pp) {
        const int j = jg + 2 * pp;
        if (j >= nchunk) break;  // short last group
        uint4 b0 = make_uint4(0u, 0u, 0u, 0u), b1 = b0;
        if (has_tok) {
          b0 = bsl[j * bstep];
          b1 = bsl[(j + 1) * bstep];
        }
        const uint32_t off = lbase + (uint32_t)(j >> 3) * boxb + ((((uint32_t)j << 4) & 0x60u) ^ hx4);
#pragma unroll
        for (int m = 0; m < M; ++m) {
          uint32_t r[4];
          ldmatrix_x4(r, off + (uint32_t)m * a.code_mat_bytes);
          // r[0]: row g chunk j, r[1]: row g+8 chunk j, r[2]: row g chunk j+1, r[3]: row g+8 chunk j+1
          const DeqWord w0 = dequant_word(r[0]), w1 = dequant_word(r[1]);
          mma_16816(d[m], w0.h04, w1.h04, w0.h15, w1.h15, b0.x, b0.y);
          mma_16816(d[m], w0.h26, w1.h26, w0.h37, w1.h37, b0.z, b0.w);
          const DeqWord w2 = dequant_word(r[2]), w3 = dequant_word(r[3]);
          mma_16816(d[m], w2.h04, w3.h04, w2.h15, w3.h15, b1.x, b1.y);
          mma_16816(d[m], w2.h26, w3.h26, w2.h37, w3.h37, b1.z, b1.w);
        }
      }
      epilogue(gi, d);
    }
  }
  const int blk = tc_red_block(NS);
  float* rw = red + (size_t)warp * M * blk;
#pragma unroll
  for (int m = 0; m < M; ++m) {
    float* rm = rw + m * blk;
    if (2 * c < NS) {
      rm[g * NS + 2 * c] = acc[m][0];
      rm[(g + 8) * NS + 2 * c] = acc[m][2];
    }
    if (2 * c + 1 < NS) {
      rm[g * NS + 2 * c + 1] = acc[m][1];
      rm[(g + 8) * NS + 2 * c + 1] = acc[m][3];
    }
  }
}

template <bool DUAL>
__device__ __forceinline__ void tc_compute(const TcGemvArgs& a, const unsigned char* sb, const uint4* Bs,
                                           const float* Cs, int ntok, int NS, float* red, int warp, int lane,
                                           const float* Xs = nullptr) {
  if (a.zp) {
    if (a.G == 32)
      tc_compute_g<DUAL, 1, true>(a, sb, Bs, Cs, Xs, ntok, NS, red, warp, lane);
    else if (a.G == 64)
      tc_compute_g<DUAL, 2, true>(a, sb, Bs, Cs, Xs, ntok, NS, red, warp, lane);
    else
      tc_compute_g<DUAL, 4, true>(a, sb, Bs, Cs, Xs, ntok, NS, red, warp, lane);
  } else if (a.G == 32) {
    tc_compute_g<DUAL, 1, false>(a, sb, Bs, Cs, Xs, ntok, NS, red, warp, lane);
  } else if (a.G == 64) {
    tc_compute_g<DUAL, 2, false>(a, sb, Bs, Cs, Xs, ntok, NS, red, warp, lane);
  } else {
    tc_compute_g<DUAL, 4, false>(a, sb, Bs, Cs, Xs, ntok, NS, red, warp, lane);
  }
}

// Outputs of an item's token tile from the K-part partials, by one warp (the
// finisher): gate/up -> h (FP16, SwiGLU), down -> y (FP32) at flat index
// perm[pos] (pos < Tk) or pos. Lane per output; the K parts are summed in
// order kp = 0 .. kparts - 1.
template <bool DUAL>
__device__ __forceinline__ void tc_finish_warp(const TcGemvArgs& a, int sgi, int rbi, int tb, int ntok, int NS,
                                               const float* red, int lane) {
  constexpr int M = DUAL ? 2 : 1;
  const int r0 = rbi * a.rb;
  const int nrows = min(a.rb, a.N - r0);
  const int pos0 = a.seg_start[sgi] + tb;
  const int kparts = a.kparts;
  const int blk = tc_red_block(NS);
  // outputs enumerated as ((u * ntok + n) * 16 + r); u = un / ntok by a
  // multiply-shift that is exact for ntok <= 8 and un < 1024
  const uint32_t inv_ntok = (65536u + (uint32_t)ntok - 1u) / (uint32_t)ntok;
  const int outputs = a.rt * 16 * ntok;
  for (int o = lane; o < outputs; o += 32) {
    const int r = o & 15, un = o >> 4;
    const int u = (int)(((uint32_t)un * inv_ntok) >> 16);
    const int n = un - u * ntok;
    const int row = u * 16 + r;
    if (row >= nrows) continue;
    const float* base = red + (size_t)u * kparts * M * blk + r * NS + n;
    float p0[kTcWarps], p1[kTcWarps];
#pragma unroll
    for (int kp = 0; kp < kTcWarps; ++kp) {
      p0[kp] = p1[kp] = 0.f;
      if (kp < kparts) {
        p0[kp] = base[(size_t)kp * M * blk];
        if (DUAL) p1[kp] = base[(size_t)(kp * M + 1) * blk];
      }
    }
    float v0 = 0.f, v1 = 0.f;
#pragma unroll
    for (int kp = 0; kp < kTcWarps; ++kp)
      if (kp < kparts) {
        v0 += p0[kp];
        v1 += p1[kp];
      }
    const int pos = pos0 + n;
    if (DUAL) {
      a.h_out[(size_t)pos * a.N + r0 + row] = __float2half_rn(silu_fast(v0) * v1);
    } else {
      const int f = (pos < a.Tk) ? a.perm[pos] : pos;
      a.y_out[(size_t)f * a.N + r0 + row] = v0;
    }
  }
}

// Hand-off of the K-part partials between the consumer warps and the
// finisher warp: two buffers used in turn (token tile ti uses buffer ti & 1);
// red_full[b] counts the consumer warps that wrote buffer b, red_free[b] is
// arrived by the finisher once it has read it.
struct TcRedBars {
  uint64_t full[2];
  uint64_t free_[2];
};
__device__ __forceinline__ void tc_red_bars_init(TcRedBars* rb) {
  for (int b = 0; b < 2; ++b) {
    mbar_init(&rb->full[b], kTcWarps);
    mbar_init(&rb->free_[b], 1);
  }
}

}  // namespace moe
