// Prefill-regime grouped W4A16 GEMM on the 5th-generation tensor cores.
//
// Horizon RunMap report, "What is implemented": the INT4 experts stay compact
// in GPU memory and run with FP16 activations; here a weight tile is expanded
// to FP16 only on chip (in tensor memory), for the MMAs that consume it.
//
// Tile = 128 MMA rows x 192 tokens of one expert segment. The weights are
// the MMA's A operand (M = 128) and the tokens its B operand (N = 192), so
// each dequantised weight row serves 192 tokens; the accumulator's TMEM lane
// is the output unit, its column the token. Gate/up tiles interleave the two
// matrices in M: row 2u is gate unit i0+u, row 2u+1 is up unit i0+u (64 units
// per tile), so SwiGLU pairs sit in adjacent lanes and meet with one shuffle.
//
// The A operand is read from tensor memory (tcgen05.mma with [a-tmem]): the
// dequantisers store each FP16 row to its TMEM lane, so shared memory carries
// only the token tiles (TMA write + MMA read) and the INT4 codes. Tensor
// memory holds two accumulator buffers (2 x 192 columns) and four A stages
// (4 x 32 columns).
//
// Warp roles of a persistent CTA (one per SM):
//   warp 0      TMA producer of the token tiles (2-D 192-row boxes of the
//               expert-sorted activations: x gathered in sorted order for
//               gate/up, h for down). A 2-D box streams at ~45 bytes per
//               SM-cycle from L2 on this part and small boxes cost about as
//               much each, so every K step is one large box.
//   warp 1      TMEM allocation and the single MMA-issuing thread
//   warps 2-9   dequantisers: codes -> (q - z) * s in FP16, one row per
//               thread, stored to the A stage in tensor memory
//   warps 10-17 epilogue: TMEM -> registers; gate/up: h = silu(g) * u -> FP16
//               h rows; down: FP32 partial rows at the pair's flat index
//   warp 18     TMA producer of the INT4 code tiles (3-D tensor map over the
//               slot pool: bytes x rows x slot; one 128-byte-wide swizzled
//               box covers four K steps)
// Rings: codes (TMA -> dequant), A (dequant -> MMA, tensor memory), B (TMA ->
// MMA), and two TMEM accumulator buffers (MMA -> epilogue), each with
// full/empty mbarriers. Every wait is bounded; a wait that gives up records
// an error, the CTA drains its in-flight copies and MMAs, frees TMEM and
// exits.
#include <cudaTypedefs.h>

#include <algorithm>

#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace moe {

namespace {

constexpr int BM = 128;  // MMA rows per tile (DUAL: 64 gate + 64 up, interleaved)
constexpr int BN = 192;  // tokens per tile
constexpr int BK = 64;   // K per pipeline step (128 bytes of FP16)
constexpr int kCodeK = 4;  // K steps per code tile: 128 bytes of codes per row, one swizzled TMA box
constexpr int kCodeStages = 4;
constexpr int kAStages = 4;  // FP16 weight tiles in tensor memory
constexpr int kBStages = 4;
constexpr int kDequantWarps = 8;
constexpr int kEpiWarps = 8;  // two per TMEM lane quadrant, each half of the columns
constexpr int kWarpProducer = 0;
constexpr int kWarpMma = 1;
constexpr int kWarpDequant0 = 2;
constexpr int kWarpEpi0 = kWarpDequant0 + kDequantWarps;
constexpr int kWarpCodes = kWarpEpi0 + kEpiWarps;  // TMA producer of the code tiles
constexpr int kGemmThreads = (kWarpCodes + 1) * 32;
constexpr int kMaxSeg = 1025;

template <bool DUAL>
struct Smem {
  static constexpr uint32_t b_tile = BN * BK * 2;      // 24 KB
  static constexpr uint32_t code_tile = BM * kCodeK * BK / 2;  // 16 KB (DUAL: 64 gate rows then 64 up rows)
  static constexpr uint32_t off_b = 0;
  static constexpr uint32_t off_codes = off_b + kBStages * b_tile;
  static constexpr uint32_t off_bar = off_codes + kCodeStages * code_tile;
  // codes_full/empty, a_full/empty, b_full/empty, acc_full/empty, drain
  static constexpr uint32_t n_bars = 2 * kCodeStages + 2 * kAStages + 2 * kBStages + 4 + 1;
  static constexpr uint32_t off_misc = off_bar + n_bars * 8;
  static constexpr uint32_t off_prefix = off_misc + 64;
  static constexpr uint32_t off_epi = off_prefix + ((kMaxSeg + 1) * 4 + 15) / 16 * 16;  // [BN] output rows of a tile
  static constexpr uint32_t bytes = off_epi + BN * 4;
  static constexpr uint32_t alloc = bytes + 1024;  // slack for 1024-byte alignment
  // tensor memory: two FP32 accumulator buffers of BN columns, then the
  // FP16 A stages (BK / 2 columns each: two K elements per column)
  static constexpr uint32_t tmem_cols = 512;
  static constexpr uint32_t acc_stride = BN;
  static constexpr uint32_t a_col0 = 2 * BN;
  static constexpr uint32_t a_cols = BK / 2;
  static constexpr int units = DUAL ? BM / 2 : BM;  // output units per tile
  static_assert(a_col0 + kAStages * a_cols <= tmem_cols, "tensor memory over-committed");
  static_assert(b_tile % 1024 == 0, "token stages must keep the 1024-byte swizzle alignment");
};

struct Bars {
  uint64_t* codes_full;
  uint64_t* codes_empty;
  uint64_t* a_full;
  uint64_t* a_empty;
  uint64_t* b_full;
  uint64_t* b_empty;
  uint64_t* acc_full;
  uint64_t* acc_empty;
  uint64_t* drain;
};

struct Misc {
  uint32_t tmem_base;
  int abort_flag;
  int total_tiles;
  int codes_issued;
  int b_issued;
  int mma_issued;
};

// barriers of the epilogue warps only (named barrier 2); the second returns
// whether any epilogue thread passed true
__device__ __forceinline__ void epi_bar() { asm volatile("bar.sync 2, %0;" ::"r"(kEpiWarps * 32) : "memory"); }
__device__ __forceinline__ bool epi_bar_any(bool v) {
  uint32_t r;
  asm volatile(
      "{ .reg .pred p, q; setp.ne.u32 p, %1, 0; bar.red.or.pred q, 2, %2, p; selp.u32 %0, 1, 0, q; }"
      : "=r"(r)
      : "r"((uint32_t)v), "r"(kEpiWarps * 32)
      : "memory");
  return r != 0;
}

// mbar_wait that adds the cycles it spent to *acc (when acc is set)
__device__ __forceinline__ bool timed_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag, uint32_t* err,
                                           unsigned long long* acc) {
  if (!acc) return mbar_wait(bar, parity, abort_flag, err);
  const long long t0 = clock64();
  const bool ok = mbar_wait(bar, parity, abort_flag, err);
  *acc += (unsigned long long)(clock64() - t0);
  return ok;
}

__device__ __forceinline__ int find_segment(const int* prefix, int nseg, int t) {
  int lo = 0, hi = nseg - 1;  // largest s with prefix[s] <= t
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (prefix[mid] <= t)
      lo = mid;
    else
      hi = mid - 1;
  }
  return lo;
}

// (q - z) * s for the 8 codes of one word (k = 8i .. 8i+7), as 8 FP16 in
// k order. Codes k=2b (low nibble) and 2b+1 (high nibble) of byte b become
// the half pair {1024 + q_lo, 1024 + q_hi} via the exponent-bias trick, then
// (h - (1024 + z)) is exact and one multiply by the FP16 scale rounds once
// (z = 8 without zero points: bias = 1032).
__device__ __forceinline__ uint4 dequant8(uint32_t w, __half2 s2, __half2 bias) {
  const uint32_t hi = w >> 4;
  uint32_t out[4];
#pragma unroll
  for (int b = 0; b < 4; ++b) {
    // byte b of w in bits 0..7, byte b of (w >> 4) in bits 16..23
    const uint32_t p = __byte_perm(w, hi, (uint32_t)(b | ((4 + b) << 8)) | 0x5400u);
    uint32_t v;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(v) : "r"(p), "r"(0x000F000Fu), "r"(0x64006400u));
    __half2 h = *reinterpret_cast<__half2*>(&v);
    h = __hmul2(__hsub2(h, bias), s2);
    out[b] = *reinterpret_cast<uint32_t*>(&h);
  }
  return make_uint4(out[0], out[1], out[2], out[3]);
}

template <bool DUAL>
__global__ void __launch_bounds__(kGemmThreads, 1)
    k_gemm(const __grid_constant__ CUtensorMap tm_codes0, const __grid_constant__ CUtensorMap tm_codes1,
           const __grid_constant__ CUtensorMap tm_act, GemmArgs a) {
  using L = Smem<DUAL>;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::off_bar);
  Bars B;
  B.codes_full = bars;
  B.codes_empty = B.codes_full + kCodeStages;
  B.a_full = B.codes_empty + kCodeStages;
  B.a_empty = B.a_full + kAStages;
  B.b_full = B.a_empty + kAStages;
  B.b_empty = B.b_full + kBStages;
  B.acc_full = B.b_empty + kBStages;
  B.acc_empty = B.acc_full + 2;
  B.drain = B.acc_empty + 2;
  Misc* misc = reinterpret_cast<Misc*>(smem + L::off_misc);
  int* prefix = reinterpret_cast<int*>(smem + L::off_prefix);

  if (tid == 0) {
    for (int i = 0; i < kCodeStages; ++i) {
      mbar_init(&B.codes_full[i], 1);
      mbar_init(&B.codes_empty[i], kDequantWarps);
    }
    for (int i = 0; i < kAStages; ++i) {
      mbar_init(&B.a_full[i], kDequantWarps / 2);
      mbar_init(&B.a_empty[i], 1);
    }
    for (int i = 0; i < kBStages; ++i) {
      mbar_init(&B.b_full[i], 1);
      mbar_init(&B.b_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&B.acc_full[i], 1);
      mbar_init(&B.acc_empty[i], kEpiWarps);
    }
    mbar_init(B.drain, 1);
    misc->abort_flag = 0;
    misc->codes_issued = 0;
    misc->b_issued = 0;
    misc->mma_issued = 0;
    fence_mbar_init();
  }
  if (warp == kWarpProducer && lane == 0) {
    prefetch_tmap(&tm_codes0);
    if (DUAL) prefetch_tmap(&tm_codes1);
    prefetch_tmap(&tm_act);
  }
  if (warp == kWarpMma) tmem_alloc(&misc->tmem_base, L::tmem_cols);
  pdl_trigger();
  pdl_wait();

  // tile prefix over the segments (segment s has m_tiles * ceil(count/BN) tiles)
  const int nseg = min(*a.num_seg, kMaxSeg);
  const int m_tiles = (a.N + L::units - 1) / L::units;
  if (warp == 0) {
    int run = 0;
    for (int base = 0; base < nseg; base += 32) {
      const int s = base + lane;
      const int c = s < nseg ? a.seg_count[s] : 0;
      int v = m_tiles * ((c + BN - 1) / BN);
      int incl = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      if (s < nseg) prefix[s] = run + incl - v;
      run += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) {
      prefix[nseg] = run;
      misc->total_tiles = run;
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const int total = misc->total_tiles;
  const uint32_t tbase = misc->tmem_base;
  unsigned long long* st_cta = a.stats ? a.stats + (size_t)blockIdx.x * kGemmStats : nullptr;
  const long long t_start = clock64();
  const int nK = a.K / BK;
  volatile int* abort_flag = &misc->abort_flag;

  if (warp == kWarpProducer) {
    // ------------------------------------------- producer of the token tiles
    if (lane == 0) {
      unsigned long long sw = 0;
      uint32_t g = 0;  // K steps over all tiles of this CTA
      bool ok = true;
      for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
        const int s = find_segment(prefix, nseg, t);
        const int local = t - prefix[s];
        const int cnt = a.seg_count[s];
        const int ntl = (cnt + BN - 1) / BN;
        const int n0 = (local % ntl) * BN;
        const int pos0 = a.seg_start[s];
        for (int kk = 0; kk < nK; ++kk, ++g) {
          const int sb = g % kBStages;
          if (!timed_wait(&B.b_empty[sb], ((g / kBStages) & 1u) ^ 1u, abort_flag, a.err, st_cta ? &sw : nullptr)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&B.b_full[sb], L::b_tile);
          tma_load_2d(smem + L::off_b + (uint32_t)sb * L::b_tile, &tm_act, kk * BK, pos0 + n0, &B.b_full[sb]);
          misc->b_issued = (int)g + 1;
        }
      }
      if (st_cta) st_cta[1] = sw;
    }
  } else if (warp == kWarpCodes) {
    // -------------------------------------------- producer of the code tiles
    if (lane == 0) {
      unsigned long long sw = 0;
      uint32_t gc = 0;  // code groups over all tiles of this CTA
      bool ok = true;
      for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
        const int s = find_segment(prefix, nseg, t);
        const int local = t - prefix[s];
        const int cnt = a.seg_count[s];
        const int ntl = (cnt + BN - 1) / BN;
        const int m0 = (local / ntl) * L::units;
        const int e = a.seg_expert[s];
        int slot = a.expert_to_slot[e];
        if (slot < 0 || slot >= a.num_slots) {
          record_error(a.err, MOE_DEV_ERR_BOUNDS);
          slot = 0;
        }
        for (int kk = 0; kk < nK; kk += kCodeK, ++gc) {
          // codes of K steps kk .. kk + kCodeK - 1: one box per matrix
          const int sc = gc % kCodeStages;
          if (!timed_wait(&B.codes_empty[sc], ((gc / kCodeStages) & 1u) ^ 1u, abort_flag, a.err,
                          st_cta ? &sw : nullptr)) {
            ok = false;
            break;
          }
          unsigned char* cdst = smem + L::off_codes + (uint32_t)sc * L::code_tile;
          mbar_arrive_expect_tx(&B.codes_full[sc], L::code_tile);
          const int cx = (kk / kCodeK) * (kCodeK * BK / 2);
          tma_load_3d(cdst, &tm_codes0, cx, m0, slot, &B.codes_full[sc]);
          if (DUAL) tma_load_3d(cdst + L::code_tile / 2, &tm_codes1, cx, m0, slot, &B.codes_full[sc]);
          misc->codes_issued = (int)gc + 1;
        }
      }
      if (st_cta) st_cta[0] = sw;
    }
  } else if (warp == kWarpMma) {
    // ----------------------------------------------------------------- MMA
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_f16_f32(BM, BN);
      unsigned long long sw[2] = {0, 0};
      uint32_t g = 0;
      int j = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < total && ok; t += gridDim.x, ++j) {
        const int ab = j & 1;
        if (!timed_wait(&B.acc_empty[ab], ((uint32_t)(j >> 1) & 1u) ^ 1u, abort_flag, a.err, st_cta ? &sw[0] : nullptr))
          break;
        tc_fence_after();
        const uint32_t d0 = tbase + (uint32_t)ab * L::acc_stride;
        for (int kk = 0; kk < nK; ++kk, ++g) {
          const int sa = g % kAStages, sb = g % kBStages;
          // one wait per K step: the dequantisers arrive on a_full only once
          // the step's token tile has landed (each waits on b_full first), so
          // a full A stage means a full token stage too. A wait in this loop
          // stalls the MMA stream (the issuing thread's queue of MMAs drains
          // meanwhile), so the loop holds as few as possible.
          if (!timed_wait(&B.a_full[sa], (g / kAStages) & 1u, abort_flag, a.err, st_cta ? &sw[1] : nullptr)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = tbase + L::a_col0 + (uint32_t)sa * L::a_cols;
          const uint32_t bb = smem_u32(smem + L::off_b + (uint32_t)sb * L::b_tile);
#pragma unroll
          for (int k16 = 0; k16 < BK / 16; ++k16) {
            const uint32_t acc = (kk > 0 || k16 > 0) ? 1u : 0u;
            mma_f16_ts(d0, a0 + k16 * 8, smem_desc_sw128(bb + k16 * 32), idesc, acc);
          }
          misc->mma_issued = 1;
          mma_commit(&B.a_empty[sa]);
          mma_commit(&B.b_empty[sb]);
        }
        if (!ok) break;
        mma_commit(&B.acc_full[ab]);
      }
      if (st_cta) {
        st_cta[2] = sw[0];
        st_cta[3] = sw[1];
      }
    }
  } else if (warp < kWarpEpi0) {
    // ------------------------------------------------------------ dequant
    // Two groups of kDequantWarps / 2 warps take alternate K steps (group
    // par takes the steps kk with kk % 2 == par), so two A stages fill at
    // once; a thread converts one A row (64 codes) per step and stores it
    // to its TMEM lane, which fixes the row: a warp reaches the lane quarter
    // warp % 4 only (the four warps of a group cover the four quarters).
    const int par = (warp - kWarpDequant0) / (kDequantWarps / 2);
    const int r = 32 * (warp & 3) + lane;  // A row 0..127 = TMEM lane
    const uint32_t a_lane = tbase + ((uint32_t)(32 * (warp & 3)) << 16) + L::a_col0;
    // A row r: DUAL -> unit r/2 of the gate (even r) or up (odd r) matrix,
    // codes row r/2 or 64 + r/2 of the stage; single -> row r.
    const int unit = DUAL ? (r >> 1) : r;
    const bool upper = DUAL && (r & 1);
    const int crow = DUAL ? ((r & 1) ? 64 + (r >> 1) : (r >> 1)) : r;
    const bool rec = st_cta && warp == kWarpDequant0 && lane == 0;
    uint32_t gbase = 0, gc = 0;  // K steps of the previous tiles, code groups (the producer's order)
    unsigned long long dw[3] = {0, 0, 0};
    bool ok = true;
    for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
      const int s = find_segment(prefix, nseg, t);
      const int local = t - prefix[s];
      const int cnt = a.seg_count[s];
      const int ntl = (cnt + BN - 1) / BN;
      const int m0 = (local / ntl) * L::units;
      const int e = a.seg_expert[s];
      int slot = a.expert_to_slot[e];
      if (slot < 0 || slot >= a.num_slots) slot = 0;
      const bool rvalid = m0 + unit < a.N;
      const uint8_t* recp = a.pool + (size_t)slot * a.record_bytes;
      const __half* sp = reinterpret_cast<const __half*>(recp + (upper ? a.s_off1 : a.s_off0)) +
                         (size_t)(m0 + unit) * a.ng;
      const uint8_t* zrow = recp + (upper ? a.z_off1 : a.z_off0) + (size_t)(m0 + unit) * a.ng;
      const int ngroups = (nK + kCodeK - 1) / kCodeK;
      // this row's scales (and zero points) for the group's next K step,
      // loaded one step ahead so their latency overlaps the current step's
      // conversion; a step of BK codes is one group, or two at G = 32 (its
      // first 32 codes in the first, the rest in the second)
      const bool two = a.G < BK;
      auto step_params = [&](int kk, uint32_t& s_pair, uint32_t& z_pair) {
        const int gi = (kk * BK) / a.G;
        const __half s0 = __ldg(sp + gi), s1 = two ? __ldg(sp + gi + 1) : s0;
        s_pair = (uint32_t)__half_as_ushort(s0) | ((uint32_t)__half_as_ushort(s1) << 16);
        uint32_t z0 = 8u, z1 = 8u;
        if (a.zp) {
          z0 = __ldg(zrow + gi);
          z1 = two ? (uint32_t)__ldg(zrow + gi + 1) : z0;
        }
        z_pair = z0 | (z1 << 16);
      };
      uint32_t sv_next = 0u, zv_next = 0x00080008u;
      if (rvalid && par < nK) step_params(par, sv_next, zv_next);
      for (int grp = 0; grp < ngroups && ok; ++grp, ++gc) {
        const int sc = gc % kCodeStages;
        int good = 1;
        if (lane == 0)
          good = timed_wait(&B.codes_full[sc], (gc / kCodeStages) & 1u, abort_flag, a.err, rec ? &dw[0] : nullptr);
        good = __shfl_sync(0xffffffffu, good, 0);
        if (!good) {
          ok = false;
          break;
        }
        const unsigned char* crowp = smem + L::off_codes + (uint32_t)sc * L::code_tile + crow * 128;
        const int k_end = min(nK, (grp + 1) * kCodeK);
        for (int kk = grp * kCodeK + par; kk < k_end; kk += 2) {
          const uint32_t g = gbase + (uint32_t)kk;
          const int sa = g % kAStages;
          const uint32_t sv = sv_next, zv = zv_next;
          if (rvalid && kk + 2 < nK) step_params(kk + 2, sv_next, zv_next);
          if (lane == 0)
            good = timed_wait(&B.a_empty[sa], ((g / kAStages) & 1u) ^ 1u, abort_flag, a.err, rec ? &dw[1] : nullptr);
          good = __shfl_sync(0xffffffffu, good, 0);
          if (!good) {
            ok = false;
            break;
          }
          tc_fence_after();
          // codes of K step kk: 16-byte chunks 2 (kk % kCodeK) and + 1 of the
          // row's 128 bytes, at their 128-byte-swizzle positions
          const int cc = (kk % kCodeK) * 2;
          const uint4 w0 = *reinterpret_cast<const uint4*>(crowp + ((cc ^ (crow & 7)) << 4));
          const uint4 w1 = *reinterpret_cast<const uint4*>(crowp + (((cc + 1) ^ (crow & 7)) << 4));
          const __half2 s_lo = __half2half2(__ushort_as_half((unsigned short)(sv & 0xFFFFu)));
          const __half2 s_hi = __half2half2(__ushort_as_half((unsigned short)(sv >> 16)));
          // 1024 + z: exponent-bias form of the zero point (exact)
          const __half2 b_lo = __half2half2(__ushort_as_half((unsigned short)(0x6400u + (zv & 0xFFFFu))));
          const __half2 b_hi = __half2half2(__ushort_as_half((unsigned short)(0x6400u + (zv >> 16))));
          const uint32_t words[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
          // columns 4c .. 4c + 3 of the row: the 8 halves of word c in k order
          uint32_t col[32];
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const uint4 q = dequant8(words[c], c < 4 ? s_lo : s_hi, c < 4 ? b_lo : b_hi);
            col[4 * c + 0] = q.x;
            col[4 * c + 1] = q.y;
            col[4 * c + 2] = q.z;
            col[4 * c + 3] = q.w;
          }
          tmem_st32(a_lane + (uint32_t)sa * L::a_cols, col);
          tmem_st_wait();
          tc_fence_before();
          // the step's token tile must have landed before the arrival
          const int sb = g % kBStages;
          if (lane == 0)
            good = timed_wait(&B.b_full[sb], (g / kBStages) & 1u, abort_flag, a.err, rec ? &dw[2] : nullptr);
          good = __shfl_sync(0xffffffffu, good, 0);
          if (!good) {
            ok = false;
            break;
          }
          if (lane == 0) mbar_arrive(&B.a_full[sa]);
        }
        if (!ok) break;
        // every dequantiser warp releases the code group once, after its steps
        __syncwarp();
        if (lane == 0) mbar_arrive(&B.codes_empty[sc]);
      }
      gbase += (uint32_t)nK;
    }
    if (st_cta && warp == kWarpDequant0 && lane == 0) {
      st_cta[4] = dw[2];
      st_cta[5] = dw[0];
      st_cta[6] = dw[1];
    }
  } else {
    // ----------------------------------------------------------- epilogue
    // Warp e of the epilogue reads TMEM lanes 32 * (warp % 4) .. + 31 (its
    // accumulator rows) and columns (BN / 2) * (e / 4) .. + BN / 2 - 1 (its
    // tokens).
    const int e = warp - kWarpEpi0, et = tid - kWarpEpi0 * 32;
    const int q = warp & 3, ch = e >> 2;
    const int row = 32 * q + lane;
    int* s_f = reinterpret_cast<int*>(smem + L::off_epi);
    unsigned long long ew = 0;
    int j = 0;
    for (int t = blockIdx.x; t < total; t += gridDim.x, ++j) {
      const int s = find_segment(prefix, nseg, t);
      const int local = t - prefix[s];
      const int cnt = a.seg_count[s];
      const int ntl = (cnt + BN - 1) / BN;
      const int m0 = (local / ntl) * L::units, n0 = (local % ntl) * BN;
      const int pos0 = a.seg_start[s];
      const int ab = j & 1;
      int good = 1;
      if (lane == 0)
        good = timed_wait(&B.acc_full[ab], (uint32_t)(j >> 1) & 1u, abort_flag, a.err,
                          (st_cta && warp == kWarpEpi0) ? &ew : nullptr);
      good = __shfl_sync(0xffffffffu, good, 0);
      if (DUAL) {
        if (!good) break;
      } else {
        // one decision for all epilogue warps (they meet at named barriers);
        // the previous tile's indices are no longer read past this point
        if (epi_bar_any(!good)) break;
        // output row (flat pair index) of every token column of the tile
        for (int c = et; c < BN; c += kEpiWarps * 32) {
          const int tok = n0 + c;
          int f = -1;
          if (tok < cnt) {
            const int pos = pos0 + tok;
            f = (pos < a.Tk) ? __ldg(a.perm + pos) : pos;
          }
          s_f[c] = f;
        }
        epi_bar();
      }
      tc_fence_after();
      // DUAL: even lanes own gate unit row/2, odd lanes its up value
      const int gunit = m0 + (DUAL ? (row >> 1) : row);
      const bool rvalid = gunit < a.N;
      const uint32_t tacc = tbase + ((uint32_t)(32 * q) << 16) + (uint32_t)ab * L::acc_stride + (BN / 2) * ch;
#pragma unroll 1
      for (int cb = 0; cb < BN / 64; ++cb) {
        uint32_t v[32];
        tmem_ld32(tacc + cb * 32, v);
        tmem_ld_wait();
        const int c0 = (BN / 2) * ch + cb * 32;
        if (DUAL) {
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            const float mine = __uint_as_float(v[c]);
            const float other = __shfl_xor_sync(0xffffffffu, mine, 1);
            const int tok = n0 + c0 + c;
            if (!(lane & 1) && rvalid && tok < cnt)
              a.h_out[(size_t)(pos0 + tok) * a.N + gunit] = __float2half_rn(silu_fast(mine) * other);
          }
        } else {
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            const int f = s_f[c0 + c];
            if (rvalid && f >= 0) a.y_out[(size_t)f * a.N + gunit] = __uint_as_float(v[c]);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&B.acc_empty[ab]);
    }
    if (st_cta && warp == kWarpEpi0 && lane == 0) st_cta[7] = ew;
  }

  // ---------------------------------------------------------------- teardown
  tc_fence_before();
  __syncthreads();
  if (st_cta && tid == 0) st_cta[8] = (unsigned long long)(clock64() - t_start);
  if (misc->abort_flag) {
    if (warp == kWarpProducer && lane == 0) {
      // let issued copies land before shared memory is released
      const int ci = misc->codes_issued, bi = misc->b_issued;
      for (int s = 0; s < kCodeStages && s < ci; ++s)
        mbar_wait(&B.codes_full[s], (uint32_t)((ci - 1 - s) / kCodeStages) & 1u, nullptr, nullptr);
      for (int s = 0; s < kBStages && s < bi; ++s)
        mbar_wait(&B.b_full[s], (uint32_t)((bi - 1 - s) / kBStages) & 1u, nullptr, nullptr);
    }
    if (warp == kWarpMma && lane == 0 && misc->mma_issued) {
      mma_commit(B.drain);
      mbar_wait(B.drain, 0, nullptr, nullptr);
    }
  }
  __syncthreads();
  tc_fence_after();
  if (warp == kWarpMma) tmem_dealloc(tbase, L::tmem_cols);
}

// Tokens in expert-sorted order for the gate/up GEMM: xs[pos] = x[perm[pos] /
// k] for pos < Tk, x[pos - Tk] for the shared expert's segment. A warp per
// row, 16-byte copies.
__global__ void __launch_bounds__(256) k_gather_rows(const __half* __restrict__ x, __half* __restrict__ xs,
                                                      const int32_t* __restrict__ perm, int Tk, int k, int rows,
                                                      int H) {
  pdl_trigger();
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int h8 = H / 8;
  for (int pos = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; pos < rows; pos += (gridDim.x * blockDim.x) >> 5) {
    const int src = pos < Tk ? __ldg(perm + pos) / k : pos - Tk;
    const uint4* in = reinterpret_cast<const uint4*>(x + (size_t)src * H);
    uint4* out = reinterpret_cast<uint4*>(xs + (size_t)pos * H);
    for (int c = lane; c < h8; c += 32) out[c] = __ldg(in + c);
  }
}

}  // namespace

cudaError_t launch_gather_rows(const __half* x, __half* xs, const int32_t* perm, int Tk, int k, int rows, int H,
                               int grid, cudaStream_t s, bool pdl) {
  return launch_ex(k_gather_rows, dim3(grid), dim3(256), 0, s, pdl, x, xs, perm, Tk, k, rows, H);
}

size_t gemm_smem_bytes(bool dual) { return dual ? Smem<true>::alloc : Smem<false>::alloc; }

cudaError_t launch_gemm(bool dual, const CUtensorMap& codes0, const CUtensorMap& codes1, const CUtensorMap& act,
                        const GemmArgs& a, int grid, cudaStream_t s, bool pdl) {
  if (dual) {
    cudaError_t e = ensure_smem(k_gemm<true>, Smem<true>::alloc);
    if (e != cudaSuccess) return e;
    return launch_ex(k_gemm<true>, dim3(grid), dim3(kGemmThreads), Smem<true>::alloc, s, pdl, codes0, codes1, act, a);
  }
  cudaError_t e = ensure_smem(k_gemm<false>, Smem<false>::alloc);
  if (e != cudaSuccess) return e;
  return launch_ex(k_gemm<false>, dim3(grid), dim3(kGemmThreads), Smem<false>::alloc, s, pdl, codes0, codes1, act, a);
}

// ---------------------------------------------------------------- tensor maps
namespace {
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}
}  // namespace

bool encode_codes_map(CUtensorMap* tm, const void* pool_section, int K, int N, int num_slots, size_t record_bytes,
                      int box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[3] = {(cuuint64_t)(K / 2), (cuuint64_t)N, (cuuint64_t)num_slots};
  const cuuint64_t strides[2] = {(cuuint64_t)(K / 2), (cuuint64_t)record_bytes};
  const cuuint32_t box[3] = {kCodeK * BK / 2, (cuuint32_t)box_rows, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(tm, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(pool_section), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_tcgemv_map(CUtensorMap* tm, const void* pool_section, int K, int N, int num_slots, size_t record_bytes,
                       int box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[3] = {(cuuint64_t)(K / 2), (cuuint64_t)N, (cuuint64_t)num_slots};
  const cuuint64_t strides[2] = {(cuuint64_t)(K / 2), (cuuint64_t)record_bytes};
  const cuuint32_t box[3] = {128, (cuuint32_t)box_rows, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(tm, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(pool_section), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_rows_map(CUtensorMap* tm, const void* base, int cols, int rows, int box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  const cuuint32_t box[2] = {BK, (cuuint32_t)box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(tm, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int gemm_tile_n() { return BN; }
int gemm_tile_k() { return BK; }

}  // namespace moe
