// Batch-1 decode: the whole layer forward of one token over a fully resident
// table in one cooperative launch, one CTA per SM.
//
// At one token the layer reads ~26 MB of expert codes (OLMoE shape) and
// does almost no arithmetic; what bounds it is how soon the bytes are
// requested and how many dependent steps follow them. Measured on this part
// (CUDA-graph replay): a launch costs ~0.7 us, the first bytes of a request
// land ~1.1 us after it is issued, and once requested the whole stream runs
// at ~7 TB/s, if it is requested in large pieces: an SM's copy engine takes
// ~60 ns per 2 KB tensor box, which caps one SM below its share of HBM, while
// 16 KB bulk copies stream at the full rate. So this kernel requests every
// byte a CTA needs in one go, in a few dozen large bulk copies, and keeps the
// chain after it short:
//   1. router logits: CTA b computes the logits of experts b, b + grid, ...
//      (16 warps, one K part each, summed in part order: the same FP32
//      arithmetic as the other small-batch paths) and publishes them; every
//      CTA counts itself and waits for all;
//   2. routing, redone in every CTA from the published logits: softmax over
//      all E, the top k by (logit descending, id ascending) in two stages
//      (the best min(k, 32) of each group of 32 ids, then the ranks among
//      those candidates), the weights and the sorted positions of the k
//      experts; CTA 0 publishes the routing once its output rows are
//      written (it is read only after the launch);
//   3. loads: work comes in units of 16 rows. The CTA's gate/up units (a
//      contiguous range of the (selected expert, intermediate row) space)
//      and, for every selected expert, its down rows (a contiguous range of
//      the output rows) are requested at once, each a contiguous block of
//      code rows copied as it lies in the record (one bulk copy per unit and
//      matrix, one per expert for the down rows), plus their scale rows;
//   4. gate/up + SwiGLU unit by unit as they land: the quantisation groups
//      are spread over 16 warps; in a group, lane (g, c) of a warp reads the
//      c-th quarter of rows g and g + 8 with 128-bit shared loads and
//      dequantises the codes in registers into mma.sync fragments (four
//      independent accumulator chains), the token's FP16 values staged in
//      the matching fragment order; the offsets are removed per group and
//      the per-group partials summed in group order; h goes to global memory
//      and the CTA counts itself done;
//   5. down: once every CTA has counted, the CTA reads all of h, computes its
//      output rows for every selected expert from the codes already in
//      shared memory and combines them (rank order, then the shared expert)
//      into its rows of the output: no further cross-CTA step.
// The two counts are epoch counters: each CTA adds one per launch (wrapping
// at a multiple of the grid), so a launch waits for the next multiple of the
// grid and nothing has to reset them. Every wait is bounded; a CTA that gives
// up records an error, still counts itself (so no CTA waits in vain) and
// lets its issued copies land before it exits.
#include "route_dev.cuh"
#include "tcgemv_dev.cuh"

namespace moe {

namespace {

constexpr int kD1Warps = 16;                     // router / routing / compute warps
constexpr int kD1Producer = kD1Warps;            // issues the copies
constexpr int kD1Threads = (kD1Warps + 1) * 32;  // 544
constexpr int kUnit = 16;                        // rows per work unit (one TMA box high)

__host__ __device__ constexpr uint32_t r16(uint32_t v) { return (v + 15u) & ~15u; }

struct D1Layout {
  uint32_t gcode, dcode, gsc, dsc, xb, xc, hb, hc, redg, redd, y, rpart, e2s, keys, cand, route, bars, ctl, total;
  uint32_t lgs, xo, wsl, sub, wstride;  // stack kernel: logits, output rows, next router slice, partial sums
  uint32_t ug, ud;  // bytes of one 16-row unit of one matrix (+ slack for the ragged last group)
  uint32_t scg, scd, ngh, ngi, nwg, nwd, ngrp, kk, ncand;
};

// Offsets from the 1024-byte aligned base of the dynamic shared memory
// (total includes the alignment slack). nwg / nwd: 8-code words of the
// token's staged fragments, a whole number of groups.
__host__ __device__ inline D1Layout d1_layout(const Decode1Args& a) {
  D1Layout L;
  const uint32_t H = (uint32_t)a.r.H, I = (uint32_t)a.I, G = (uint32_t)a.G, E = (uint32_t)a.r.E;
  const uint32_t k = (uint32_t)a.r.k, ns = (uint32_t)a.nseg_max;
  const uint32_t mug = (uint32_t)a.max_units_g, mud = (uint32_t)a.max_units_d;
  L.ngh = (H + G - 1) / G;
  L.ngi = (I + G - 1) / G;
  L.nwg = L.ngh * (G / 8u);
  L.nwd = L.ngi * (G / 8u);
  // a lane of the ragged last group may read up to G/2 bytes past a row
  L.ug = r16((uint32_t)kUnit * (H / 2u) + G / 2u);
  L.ud = r16(mud * (uint32_t)kUnit * (I / 2u) + G / 2u);  // all of a segment's down rows
  L.scg = (uint32_t)kUnit * L.ngh * 2u;
  L.scd = (uint32_t)kUnit * L.ngi * 2u;
  L.kk = k < 32u ? k : 32u;
  L.ngrp = (E + 31u) / 32u;
  L.ncand = L.ngrp * L.kk;
  uint32_t o = 0;
  L.gcode = o;  // [unit][gate, up] rows
  o += mug * 2u * L.ug;
  L.dcode = o;  // [segment] rows
  o += ns * L.ud;
  L.gsc = o;
  o += r16(mug * 2u * L.scg);
  L.dsc = o;
  o += r16(ns * mud * L.scd);
  L.xb = o;
  o += L.nwg * 16u;
  L.xc = o;
  o += r16(L.ngh * 4u);
  // per-warp scratch of the down phase (the h words of four groups in
  // fragment order): the gate/up code rows once those are consumed
  const uint32_t hb_bytes = (uint32_t)kD1Warps * 4u * (G / 8u) * 16u;
  if (hb_bytes <= mug * 2u * L.ug) {
    L.hb = L.gcode;
  } else {
    L.hb = o;
    o += hb_bytes;
  }
  L.hc = L.hb;
  L.redg = o;
  o += mug * L.ngh * 2u * kUnit * 4u;
  // stack kernel: the 8 partial-logit subtotals of every expert live in the
  // gate/up reduction area (free at the start of a layer) when they fit
  L.sub = L.redg;
  if (a.stack && 8u * E * 4u > mug * L.ngh * 2u * kUnit * 4u) {
    L.sub = o;
    o += 8u * E * 4u;
  }
  L.redd = o;  // down partials
  o += mud * ns * L.ngi * kUnit * 4u;
  L.y = o;
  o += ns * mud * kUnit * 4u;
  L.rpart = o;
  o += (uint32_t)a.max_rows_rt * kLogitParts * 4u;
  L.e2s = o;
  o += r16((E + 1u) * 4u);
  L.keys = o;
  o += L.ngrp * 32u * 4u;
  L.cand = o;  // keys then ids, each padded to a multiple of 4 entries
  o += r16(((L.ncand + 3u) & ~3u) * 8u);
  L.route = o;
  o += r16((4u * k + 2u * ns + 8u + 3u * mug) * 4u);
  L.bars = o;
  o += (mug + ns) * 8u;
  L.ctl = o;
  o += 64u;
  L.wstride = mud * (uint32_t)kUnit;  // floats per expert in the router slice
  o = r16(o);  // the router slice takes 16-byte asynchronous copies
  L.lgs = L.xo = L.wsl = o;
  if (a.stack) {
    L.lgs = o;
    o += r16(E * 4u);
    L.xo = o;
    o += L.wstride * 4u;
    L.wsl = o;
    o += E * L.wstride * 4u;
  }
  L.total = o + 1024u;  // alignment slack of the base
  return L;
}

// Partial p (of kLogitParts) of expert e's logit for the one token: the
// lane-strided FP32 FMA chain and butterfly of warp_logit_partial, so the
// logits are bit-identical to the other small-batch paths'.
__device__ __forceinline__ float logit_part_t1(const RouteArgs& a, int e, int p) {
  const int lane = threadIdx.x & 31;
  const int H = a.H;
  const int h4b = (p * (H / 4)) / kLogitParts, h4e = ((p + 1) * (H / 4)) / kLogitParts;
  float acc = 0.f;
  const float4* wr4 = reinterpret_cast<const float4*>(a.wr + (size_t)e * H) + h4b;
  const uint2* x2 = reinterpret_cast<const uint2*>(a.x) + h4b;
#pragma unroll 2
  for (int h4 = lane; h4 < h4e - h4b; h4 += 32) {
    const float4 wv = __ldg(wr4 + h4);
    const uint2 raw = __ldg(x2 + h4);
    const float2 x01 = __half22float2(*reinterpret_cast<const __half2*>(&raw.x));
    const float2 x23 = __half22float2(*reinterpret_cast<const __half2*>(&raw.y));
    acc = fmaf(wv.x, x01.x, acc);
    acc = fmaf(wv.y, x01.y, acc);
    acc = fmaf(wv.z, x23.x, acc);
    acc = fmaf(wv.w, x23.y, acc);
  }
  return warp_sum(acc);
}

// (h0, h4), (h1, h5), (h2, h6), (h3, h7) of eight consecutive halves: the B
// fragment order of one 32-bit code word (see tcgemv_dev.cuh).
__device__ __forceinline__ uint4 b_frag(uint4 v) {
  uint4 o;
  o.x = __byte_perm(v.x, v.z, 0x5410);
  o.y = __byte_perm(v.x, v.z, 0x7632);
  o.z = __byte_perm(v.y, v.w, 0x5410);
  o.w = __byte_perm(v.y, v.w, 0x7632);
  return o;
}

// MMA sums of NG consecutive quantisation groups gi0 .. gi0 + NG - 1 of a
// 16-row unit stored row-major (R bytes per row) for M matrices (mstride
// bytes apart), for one token (the lanes of fragment column 0 hold it, the
// rest multiply zeros). Lane (g, c) reads CPG 8-code words of rows g and
// g + 8 at byte gi * G/2 + c * CPG * 4 (one 128- or 64-bit shared load per
// row and group), so one k16 step pairs word t of every lane; its B fragment
// is the staged token word at the same index (frag: the token's staged
// words from group gi0 on, G/8 per group). All loads are issued before the
// first MMA; every
// (group, matrix) has its own accumulator chain.
template <int M, int CPG, int NG>
__device__ __forceinline__ void quad_groups_mma(float (&D)[NG][M][4], const unsigned char* unit, uint32_t R,
                                                uint32_t mstride, int gi0, int g, int c, const uint4* frag,
                                                bool has_tok) {
  uint32_t lo[NG][M][CPG], hi[NG][M][CPG];
#pragma unroll
  for (int n = 0; n < NG; ++n)
#pragma unroll
    for (int m = 0; m < M; ++m) {
      const unsigned char* p0 = unit + (size_t)m * mstride + (size_t)g * R + (size_t)(gi0 + n) * (CPG * 16) +
                                (size_t)c * (CPG * 4);
      const unsigned char* p1 = p0 + (size_t)8 * R;
      if constexpr (CPG == 4) {
        const uint4 v0 = *reinterpret_cast<const uint4*>(p0), v1 = *reinterpret_cast<const uint4*>(p1);
        lo[n][m][0] = v0.x, lo[n][m][1] = v0.y, lo[n][m][2] = v0.z, lo[n][m][3] = v0.w;
        hi[n][m][0] = v1.x, hi[n][m][1] = v1.y, hi[n][m][2] = v1.z, hi[n][m][3] = v1.w;
      } else {
        const uint2 v0 = *reinterpret_cast<const uint2*>(p0), v1 = *reinterpret_cast<const uint2*>(p1);
        lo[n][m][0] = v0.x, lo[n][m][1] = v0.y;
        hi[n][m][0] = v1.x, hi[n][m][1] = v1.y;
      }
    }
#pragma unroll
  for (int n = 0; n < NG; ++n)
#pragma unroll
    for (int m = 0; m < M; ++m)
#pragma unroll
      for (int i = 0; i < 4; ++i) D[n][m][i] = 0.f;
#pragma unroll
  for (int n = 0; n < NG; ++n)
#pragma unroll
    for (int t = 0; t < CPG; ++t) {
      const uint4 b = has_tok ? frag[n * (4 * CPG) + c * CPG + t] : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
      for (int m = 0; m < M; ++m) {
        const DeqWord wl = dequant_word(lo[n][m][t]), wh = dequant_word(hi[n][m][t]);
        mma_16816(D[n][m], wl.h04, wh.h04, wl.h15, wh.h15, b.x, b.y);
        mma_16816(D[n][m], wl.h26, wh.h26, wl.h37, wh.h37, b.z, b.w);
      }
    }
}

// (sum of even, sum of odd) halves of one 8-half token word, paired as the
// B fragment pairs them: (x0 + x4) + (x2 + x6), (x1 + x5) + (x3 + x7).
__device__ __forceinline__ float2 word_sums(uint4 v) {
  const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&v.x));  // x0, x1
  const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&v.y));  // x2, x3
  const float2 c = __half22float2(*reinterpret_cast<const __half2*>(&v.z));  // x4, x5
  const float2 d = __half22float2(*reinterpret_cast<const __half2*>(&v.w));  // x6, x7
  return make_float2((a.x + c.x) + (b.x + d.x), (a.y + c.y) + (b.y + d.y));
}

// Group constant 1032 sum_even + 72 sum_odd of the staged token words
// [w0, w0 + n): word by word, then pairs (the constant the offsets of the
// codes (1024 + q) / (64 + q) leave in a group's MMA sum).
__device__ __forceinline__ float words_const(const uint4* frag, int w0, int n) {
  float se = 0.f, so = 0.f;
  for (int w = w0; w < w0 + n; ++w) {
    const uint4 o = frag[w];
    const float2 p0 = __half22float2(*reinterpret_cast<const __half2*>(&o.x));
    const float2 p1 = __half22float2(*reinterpret_cast<const __half2*>(&o.y));
    const float2 p2 = __half22float2(*reinterpret_cast<const __half2*>(&o.z));
    const float2 p3 = __half22float2(*reinterpret_cast<const __half2*>(&o.w));
    se += (p0.x + p0.y) + (p2.x + p2.y);
    so += (p1.x + p1.y) + (p3.x + p3.y);
  }
  return 1032.f * se + 72.f * so;
}

// Epoch counters: arrive once per launch (wrapping increment), and wait until
// all `grid` CTAs of this launch have arrived, given the value read before
// this CTA's own arrival.
__device__ __forceinline__ void epoch_arrive(uint32_t* p, uint32_t mod) {
  asm volatile("red.release.gpu.global.inc.u32 [%0], %1;" ::"l"(p), "r"(mod - 1u) : "memory");
}
__device__ __forceinline__ uint32_t ld_relaxed(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ bool epoch_reached(uint32_t cur, uint32_t base, uint32_t mod, uint32_t grid) {
  return (cur + mod - base) % mod >= grid;
}
__device__ __forceinline__ bool epoch_wait(const uint32_t* p, uint32_t base, uint32_t mod, uint32_t grid,
                                           volatile int* abort_flag, uint32_t* err) {
  if (epoch_reached(ld_acquire(p), base, mod, grid)) return true;
  const long long t0 = clock64();
  while (true) {
    __nanosleep(32);
    if (epoch_reached(ld_acquire(p), base, mod, grid)) return true;
    if (*abort_flag) return false;
    if (clock64() - t0 > kSpinLimitCycles) {
      record_error(err, MOE_DEV_ERR_TIMEOUT);
      *abort_flag = 1;
      return false;
    }
  }
}

// Gate/up tiles of a CTA whose rows are the 8-row granules [g0, g1) of the
// (segment, intermediate row) space, gpe granules per expert: 16 rows, or 8
// at the end of an expert's piece. Tile t (< 0: none) is written to *s, *r0
// (row inside the expert) and *n; returns the number of tiles.
__host__ __device__ inline int walk_tiles(int g0, int g1, int gpe, int t, int* s, int* r0, int* n) {
  int cur = g0, i = 0;
  while (cur < g1) {
    const int sq = cur / gpe;
    const int pend = g1 < (sq + 1) * gpe ? g1 : (sq + 1) * gpe;
    const int n8 = pend - cur < 2 ? pend - cur : 2;
    if (i == t) {
      *s = sq;
      *r0 = (cur - sq * gpe) * 8;
      *n = n8 * 8;
    }
    cur += n8;
    ++i;
  }
  return i;
}

// part[e] = sum over the CTA's output rows r of xo[r] * w[e * ws + r], one
// expert per thread, the rows taken from (e / 2) on (so that, at 16 rows a
// slice, the 32 lanes of a warp read 32 different banks); zero without rows.
__device__ __forceinline__ void d1_row_partials(const float* xo, const float* w, int ws, int E, int ndr,
                                                float* part) {
  for (int e = threadIdx.x; e < E; e += kD1Threads) {
    float acc = 0.f;
    int r = ndr > 0 ? (e >> 1) % ndr : 0;
    for (int i = 0; i < ndr; ++i) {
      acc = fmaf(xo[r], w[e * ws + r], acc);
      r = r + 1 == ndr ? 0 : r + 1;
    }
    part[e] = acc;
  }
}

constexpr int kD1Runs = 8;       // stack kernel: runs of CTAs the partial logits are summed in
constexpr int kD1RunMax = 32;    // most CTAs in a run (grid <= 256)

// One layer of the batch-1 decode. STACK: the layer runs inside the stack
// kernel (its logits come from the partials the CTAs published at the end of
// the layer before; at its end it publishes the next layer's).
template <int NV, int CPG, bool STACK>
__device__ __forceinline__ void d1_layer(const Decode1Args& a, unsigned char* smem, const D1Layout& L, int layer,
                                         bool traced) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int H = a.r.H, I = a.I, E = a.r.E, k = a.r.k;
  const int grid = gridDim.x, bid = blockIdx.x;
  const int nseg = k + a.r.has_shared;
  const int mug = a.max_units_g, ns_max = a.nseg_max;
  // gate/up rows: 8-row granules of the (segment, row) space, split evenly
  // over the CTAs and cut into tiles of 16 rows (8 at an expert's end)
  const int gpe = I / 8;
  const int g0 = (int)((long long)bid * nseg * gpe / grid), g1 = (int)((long long)(bid + 1) * nseg * gpe / grid);
  int nu;
  {
    int ds0, ds1, ds2;
    nu = walk_tiles(g0, g1, gpe, -1, &ds0, &ds1, &ds2);
  }
  const int d0 = (int)((long long)bid * (H / kUnit) / grid), ndu = (int)((long long)(bid + 1) * (H / kUnit) / grid) - d0;
  const int ndr = ndu * kUnit;  // down rows of this CTA
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L.bars);  // [mug] gate/up units, then [ns_max] segments
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L.ctl);
  int* issued = reinterpret_cast<int*>(smem + L.ctl + 4);
  float* s_stat = reinterpret_cast<float*>(smem + L.ctl + 8);       // softmax max, denominator
  uint32_t* s_base = reinterpret_cast<uint32_t*>(smem + L.ctl + 16);  // epoch bases
  int32_t* e2s = reinterpret_cast<int32_t*>(smem + L.e2s);
  int32_t* route = reinterpret_cast<int32_t*>(smem + L.route);
  int32_t* sel_id = route;                               // [k] rank order
  float* sel_key = reinterpret_cast<float*>(route + k);  // [k]
  float* sel_w = reinterpret_cast<float*>(route + 2 * k);
  int32_t* pos_of_rank = route + 3 * k;  // [k]
  int32_t* seg_expert = route + 4 * k;   // [ns_max]
  int32_t* seg_slot = seg_expert + ns_max;
  int32_t* tile_s = seg_slot + ns_max;  // [mug] gate/up tiles: segment, first row, rows
  int32_t* tile_r0 = tile_s + mug;
  int32_t* tile_n = tile_r0 + mug;
  uint32_t* logits_ready = a.ctr;
  uint32_t* gu_done = a.ctr + 1;
  const uint32_t mod = a.ctr_mod;
  unsigned long long* const tb = traced ? a.trace : nullptr;
  unsigned long long* tr = (tid == 0) ? tb : nullptr;
  unsigned long long* trp = (tid == kD1Producer * 32) ? tb : nullptr;
  unsigned long long* trw = (tid == (kD1Warps - 1) * 32) ? tb : nullptr;  // last consumer warp

  // Every barrier in use completes one phase per layer (the layers of a stack
  // have one shape, so a CTA has the same tiles in each): layer l waits for
  // the phase of parity l & 1; they are initialised once.
  const uint32_t par = (uint32_t)layer & 1u;
  trace_mark(tr, 0);
  if (layer == 0) {
    if (tid == 0) {
      for (int i = 0; i < mug + ns_max; ++i) mbar_init(&bars[i], 1);
      *issued = 0;
      fence_mbar_init();
    }
    if (!STACK) {
      // Inputs that no earlier launch writes (the router rows, the slot map)
      // and the tile list are requested / built before the wait on the
      // previous launch, so their latency overlaps its tail.
      const int rows0 = bid < E ? (E - 1 - bid) / grid + 1 : 0;
      const int lines = H / 32;  // 128-byte lines of one FP32 router row
      for (int q = tid; q < rows0 * lines; q += kD1Threads)
        prefetch_l2(a.r.wr + (size_t)(bid + (q / lines) * grid) * H + (size_t)(q % lines) * 32);
      if (warp == kD1Producer) {
        if (lane == 0)
          for (int cur = g0, t = 0; cur < g1 && t < mug; ++t) {
            const int sq = cur / gpe;
            const int pend = min(g1, (sq + 1) * gpe);
            const int n8 = min(2, pend - cur);
            tile_s[t] = sq;
            tile_r0[t] = (cur - sq * gpe) * 8;
            tile_n[t] = n8 * 8;
            cur += n8;
          }
        for (int e = lane; e < E + a.r.has_shared; e += 32) e2s[e] = __ldg(a.expert_to_slot + e);
      }
    }
    // programmatic dependent launch: nothing above wrote global memory
    pdl_trigger();
    pdl_wait();
    __syncthreads();
  } else if (tid == 0) {
    *issued = 0;  // read by tid 0 alone (teardown), after the block syncs below
  }
  trace_mark(tr, 1);

  // ------------------------------------------------ 1. router logits (FP32)
  const int my_rows = bid < E ? (E - 1 - bid) / grid + 1 : 0;
  float* rpart = reinterpret_cast<float*>(smem + L.rpart);
  uint4* xb = reinterpret_cast<uint4*>(smem + L.xb);
  float* xc = reinterpret_cast<float*>(smem + L.xc);
  const int nwg = (int)L.nwg, wpg = a.G / 8;  // staged words, words per group
  float* lgs = reinterpret_cast<float*>(smem + L.lgs);  // stack kernel: this layer's logits
  float* xo = reinterpret_cast<float*>(smem + L.xo);    // stack kernel: the CTA's output rows
  float* wsl = reinterpret_cast<float*>(smem + L.wsl);  // stack kernel: router slice of those rows
  const int wst = (int)L.wstride;
  if constexpr (STACK) {
    const int d0r = d0 * kUnit;
    if (layer == 0) {
      if (tid == 0) {
        // epoch bases of the launch, read before this CTA's first arrival
        s_base[0] = ld_relaxed(logits_ready);
        s_base[1] = ld_relaxed(gu_done);
      }
      // the first layer's partial logits over the CTA's rows of its input
      // (those of later layers are formed at the end of the layer before)
      for (int q = tid; q < E * ndr; q += kD1Threads) {
        const int e = q / ndr, r = q - e * ndr;
        wsl[e * wst + r] = __ldg(a.r.wr + (size_t)e * H + d0r + r);
      }
      for (int r = tid; r < ndr; r += kD1Threads) xo[r] = __half2float(a.r.x[d0r + r]);
      __syncthreads();
      d1_row_partials(xo, wsl, wst, E, ndr, a.part_in + (size_t)bid * E);
      __syncthreads();
      if (tid == 0) epoch_arrive(logits_ready, mod);
    }
    if (warp == kD1Producer) {
      if (lane == 0) {
        for (int cur = g0, t = 0; cur < g1 && t < mug; ++t) {
          const int sq = cur / gpe;
          const int pend = min(g1, (sq + 1) * gpe);
          const int n8 = min(2, pend - cur);
          tile_s[t] = sq;
          tile_r0[t] = (cur - sq * gpe) * 8;
          tile_n[t] = n8 * 8;
          cur += n8;
        }
        if (nu > mug) {
          record_error(a.r.err, MOE_DEV_ERR_BOUNDS);
          *abort_flag = 1;
        }
      }
      for (int e = lane; e < E + a.r.has_shared; e += 32) e2s[e] = __ldg(a.expert_to_slot + e);
    } else if (tid == 0) {
      // every CTA has published this layer's partials (and so its rows of
      // this layer's input)
      const uint32_t base = (s_base[0] - s_base[0] % (uint32_t)grid + (uint32_t)layer * (uint32_t)grid) % mod;
      epoch_wait(logits_ready, base, mod, (uint32_t)grid, abort_flag, a.r.err);
      trace_mark(tr, 3);
    }
    __syncthreads();
    float* sub = reinterpret_cast<float*>(smem + L.sub);
    // The input (written by every CTA during this launch: L2 loads) and the
    // partial logits, summed in a fixed order: kD1Runs runs of consecutive
    // CTAs, each run in CTA order, then the runs in order, then the bias. A
    // thread issues its partials' loads and its input word's load before it
    // uses either, so all of them are in flight at once.
    const uint4* xg = reinterpret_cast<const uint4*>(a.r.x);
    for (int q0 = 0; q0 < max(nwg, kD1Runs * E); q0 += kD1Threads) {
      const int q = q0 + tid;
      const bool has_p = q < kD1Runs * E, has_x = q < nwg;
      const int c = has_p ? q / E : 0, e = has_p ? q - c * E : 0;
      const int b0 = c * grid / kD1Runs, n = has_p ? (c + 1) * grid / kD1Runs - b0 : 0;
      float t[kD1RunMax];
#pragma unroll
      for (int i = 0; i < kD1RunMax; ++i) t[i] = i < n ? __ldcg(a.part_in + (size_t)(b0 + i) * E + e) : 0.f;
      const uint4 xv = (has_x && 8 * q < H) ? __ldcg(xg + q) : make_uint4(0u, 0u, 0u, 0u);
      if (has_p) {
        float v = 0.f;
#pragma unroll
        for (int i = 0; i < kD1RunMax; ++i)
          if (i < n) v += t[i];
        sub[c * E + e] = v;
      }
      if (has_x) xb[q] = b_frag(xv);
    }
    __syncthreads();
    trace_mark(tr, 2);
    for (int q = tid; q < E + (int)L.ngh; q += kD1Threads) {
      if (q < E) {
        float v = sub[q];
        for (int c = 1; c < kD1Runs; ++c) v += sub[c * E + q];
        lgs[q] = v + (a.r.bias ? __ldg(a.r.bias + q) : 0.f);
      } else {
        xc[q - E] = words_const(xb, (q - E) * wpg, wpg);
      }
    }
    __syncthreads();
  } else {
  if (warp < kD1Warps) {
    for (int i = 0; i < my_rows; ++i) {
      const float v = logit_part_t1(a.r, bid + i * grid, warp);
      if (lane == 0) rpart[i * kLogitParts + warp] = v;
    }
  } else {
    // epoch bases (read before this CTA arrives; the slot map and the tile
    // list were built before the wait), the token's words in fragment order
    // (zero past H)
    if (lane == 0) {
      s_base[0] = ld_relaxed(logits_ready);
      s_base[1] = ld_relaxed(gu_done);
      if (nu > mug) {
        record_error(a.r.err, MOE_DEV_ERR_BOUNDS);
        *abort_flag = 1;
      }
    }
    for (int w = lane; w < nwg; w += 32)
      xb[w] = 8 * w < H ? b_frag(__ldg(reinterpret_cast<const uint4*>(a.r.x) + w)) : make_uint4(0u, 0u, 0u, 0u);
  }
  __syncthreads();
  if (tid == 0) {
    for (int i = 0; i < my_rows; ++i) {
      const int e = bid + i * grid;
      float v = 0.f;
      for (int p = 0; p < kLogitParts; ++p) v += rpart[i * kLogitParts + p];
      a.r.logits[e] = v + (a.r.bias ? __ldg(a.r.bias + e) : 0.f);
    }
    // every CTA counts itself once; the release orders its logits before it
    const uint32_t base = s_base[0] - s_base[0] % (uint32_t)grid;
    epoch_arrive(logits_ready, mod);
    trace_mark(tr, 2);
    epoch_wait(logits_ready, base, mod, (uint32_t)grid, abort_flag, a.r.err);
    trace_mark(tr, 3);
  } else if (tid >= 32) {
    for (int gi = tid - 32; gi < (int)L.ngh; gi += kD1Threads - 32) xc[gi] = words_const(xb, gi * wpg, wpg);
  }
  __syncthreads();
  }  // !STACK

  // ------------------------------------------------------------ 2. routing
  const int ngrp = (int)L.ngrp, kk = (int)L.kk, ncand = (int)L.ncand, ncand4 = (ncand + 3) & ~3;
  float* keys = reinterpret_cast<float*>(smem + L.keys);
  float* cand_key = reinterpret_cast<float*>(smem + L.cand);
  int32_t* cand_id = reinterpret_cast<int32_t*>(cand_key + ncand4);
  // Ranks are counted against values read back from shared memory as
  // broadcast 128-bit loads: on this part a warp's shuffles run one after
  // another at ~30 cycles each, shared loads overlap.
  if (warp < kD1Warps) {
    if (warp == 0 && lane < ncand4 - ncand) {
      cand_key[ncand + lane] = -INFINITY;  // padding that never ranks ahead
      cand_id[ncand + lane] = 0x7fffffff;
    }
    // stage 1: the best kk of each group of 32 consecutive ids (rank inside
    // the group by key descending, id ascending; ids past E are -inf
    // sentinels that lose every tie)
    for (int gq = warp; gq < ngrp; gq += kD1Warps) {
      const int e = gq * 32 + lane;
      const float v = e < E ? route_key(STACK ? lgs[e] : __ldcg(a.r.logits + e)) : -INFINITY;
      keys[e] = v;
      __syncwarp();
      const float4* k4 = reinterpret_cast<const float4*>(keys + gq * 32);
      int r = 0;
#pragma unroll
      for (int o4 = 0; o4 < 8; ++o4) {
        const float4 ov = k4[o4];
        const int o = 4 * o4;
        r += (ov.x > v || (ov.x == v && o + 0 < lane)) ? 1 : 0;
        r += (ov.y > v || (ov.y == v && o + 1 < lane)) ? 1 : 0;
        r += (ov.z > v || (ov.z == v && o + 2 < lane)) ? 1 : 0;
        r += (ov.w > v || (ov.w == v && o + 3 < lane)) ? 1 : 0;
      }
      if (r < kk) {
        cand_key[gq * kk + r] = v;
        cand_id[gq * kk + r] = e;
      }
    }
  } else {
    // softmax maximum and denominator, the summation of warp_softmax_topk
    float v[NV];
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      const int e = lane + 32 * i;
      v[i] = e < E ? route_key(STACK ? lgs[e] : __ldcg(a.r.logits + e)) : -INFINITY;
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
    if (lane == 0) {
      s_stat[0] = m;
      s_stat[1] = ssum;
    }
  }
  __syncthreads();
  trace_mark(tr, 4);
  // stage 2: ranks among the candidates; ranks 0..k-1 are the selection.
  // Few candidates: the producer warp alone, so that it goes on to issue the
  // copies without another block-wide step; many: the whole CTA.
  const bool warp_stage2 = ncand <= 64;
  if (!warp_stage2) {
    const float4* k4 = reinterpret_cast<const float4*>(cand_key);
    const int4* i4 = reinterpret_cast<const int4*>(cand_id);
    for (int c = tid; c < ncand; c += kD1Threads) {
      const float v = cand_key[c];
      const int id = cand_id[c];
      int r = 0;
      for (int q4 = 0; q4 < ncand4 / 4; ++q4) {
        const float4 ov = k4[q4];
        const int4 oi = i4[q4];
        r += (ov.x > v || (ov.x == v && oi.x < id)) ? 1 : 0;
        r += (ov.y > v || (ov.y == v && oi.y < id)) ? 1 : 0;
        r += (ov.z > v || (ov.z == v && oi.z < id)) ? 1 : 0;
        r += (ov.w > v || (ov.w == v && oi.w < id)) ? 1 : 0;
      }
      if (r < k) {
        sel_id[r] = id;
        sel_key[r] = v;
      }
    }
    __syncthreads();
  }
  unsigned char* gcode = smem + L.gcode;
  unsigned char* dcode = smem + L.dcode;
  const uint32_t rowg = (uint32_t)H / 2u, rowd = (uint32_t)I / 2u;
  if (warp == kD1Producer) {
    if (warp_stage2) {
      // one or two candidates per lane, ranked against all of them
      const float4* k4 = reinterpret_cast<const float4*>(cand_key);
      const int4* i4 = reinterpret_cast<const int4*>(cand_id);
      for (int c = lane; c < ncand; c += 32) {
        const float v = cand_key[c];
        const int id = cand_id[c];
        int r = 0;
        for (int q4 = 0; q4 < ncand4 / 4; ++q4) {
          const float4 ov = k4[q4];
          const int4 oi = i4[q4];
          r += (ov.x > v || (ov.x == v && oi.x < id)) ? 1 : 0;
          r += (ov.y > v || (ov.y == v && oi.y < id)) ? 1 : 0;
          r += (ov.z > v || (ov.z == v && oi.z < id)) ? 1 : 0;
          r += (ov.w > v || (ov.w == v && oi.w < id)) ? 1 : 0;
        }
        if (r < k) {
          sel_id[r] = id;
          sel_key[r] = v;
        }
      }
      __syncwarp();
    }
    if (lane == 0) trace_mark(trp, 5);
    // sorted positions (ascending expert id) and slots first: the copies
    // need them; the weights after the copies are on their way
    int my_id = 0, pos = 0;
    if (lane < k) {
      my_id = sel_id[lane];
      for (int j = 0; j < k; ++j) pos += sel_id[j] < my_id ? 1 : 0;
      pos_of_rank[lane] = pos;
      seg_expert[pos] = my_id;
    }
    __syncwarp();
    if (lane == 0 && a.r.has_shared) seg_expert[k] = E;
    __syncwarp();
    int bad = 0;
    if (lane < nseg) {
      const int sl = e2s[seg_expert[lane]];
      bad = (sl < 0 || sl >= a.num_slots) ? 1 : 0;
      seg_slot[lane] = sl;
    }
    if (__any_sync(0xffffffffu, bad) && lane == 0) {
      record_error(a.r.err, MOE_DEV_ERR_BOUNDS);
      *abort_flag = 1;
    }
    __syncwarp();
    // the consumers may go on (their scale rows, then the units as they land)
    asm volatile("bar.arrive 2, %0;" ::"n"(kD1Threads) : "memory");
    // ----------------------------------------------------------- 3. loads
    const bool go = __shfl_sync(0xffffffffu, *abort_flag ? 0 : 1, 0);
    const uint64_t pol = l2_policy_evict_first();
    if (go && lane == 0) {
      // from one lane, tile by tile: the copy engine serves requests in
      // order, so the first tile lands (and its compute starts) first
      for (int u = 0; u < nu; ++u) {
        const int sq = tile_s[u], r0 = tile_r0[u];
        const uint32_t nb = (uint32_t)tile_n[u] * rowg;
        const uint8_t* rec = a.pool + (size_t)seg_slot[sq] * a.record_bytes;
        mbar_arrive_expect_tx(&bars[u], 2u * nb);
        unsigned char* dst = gcode + (size_t)u * 2u * L.ug;
        bulk_g2s(dst, rec + a.off_q[0] + (size_t)r0 * rowg, nb, &bars[u], pol);
        bulk_g2s(dst + L.ug, rec + a.off_q[1] + (size_t)r0 * rowg, nb, &bars[u], pol);
      }
      *issued = 1;
      trace_mark(trp, 6);
    }
    __syncwarp();
    if (go && lane == 0) {
      // the down rows once this CTA's gate/up rows have landed: until then
      // the gate/up bytes of every CTA have HBM to themselves
      // (after a failed wait every down barrier is still armed, with no
      // bytes, so that the teardown's waits end)
      bool landed = true;
      for (int u = 0; u < nu && landed; ++u) landed = mbar_wait_sleep(&bars[u], par, abort_flag, a.r.err);
      for (int sq = 0; sq < ns_max; ++sq) {
        uint64_t* bar = &bars[mug + sq];
        const bool any = landed && sq < nseg && ndr > 0;
        mbar_arrive_expect_tx(bar, any ? (uint32_t)ndr * rowd : 0u);
        if (!any) continue;
        const uint8_t* rec = a.pool + (size_t)seg_slot[sq] * a.record_bytes;
        bulk_g2s(dcode + (size_t)sq * L.ud, rec + a.off_q[2] + (size_t)d0 * kUnit * rowd, (uint32_t)ndr * rowd, bar,
                 pol);
      }
      trace_mark(trp, 8);
    }
    // weights (rank order): p = exp(l - max) / denominator, summed in rank order
    const float m = s_stat[0], ssum = s_stat[1];
    float my_p = 0.f;
    if (lane < k) my_p = expf(sel_key[lane] - m) / ssum;
    // the selected probabilities summed in rank order (as warp_softmax_topk)
    if (lane < k) sel_w[lane] = my_p;
    __syncwarp();
    float psel = 0.f;
    for (int j = 0; j < k; ++j) psel += sel_w[j];
    __syncwarp();
    if (lane < k) sel_w[lane] = a.r.renorm ? my_p / psel : my_p;
    __syncwarp();
    if (lane == 0) trace_mark(trp, 7);
  } else {
    // consumers: parked (no issue slots taken) until the gate/up copies are
    // issued, then the scale rows by plain loads
    asm volatile("bar.sync 2, %0;" ::"n"(kD1Threads) : "memory");
    if (!*abort_flag) {
      // asynchronous 16-byte copies: in flight with the code copies, waited
      // for (cp.async.wait_all + a consumer barrier) before the first use
      const int ngs = (int)(L.scg / 16u), nds = ndu * (int)(L.scd / 16u);
      const int n_g = nu * 2 * ngs, n_all = n_g + nseg * nds;
      // stack kernel: the next layer's router slice of this CTA's output
      // rows, for the partial logits it forms at the end of this layer
      const int cpe = ndr / 4, n_w = (STACK && a.wr_next) ? E * cpe : 0;
      for (int q = tid; q < n_all + n_w; q += kD1Warps * 32) {
        const uint8_t* src;
        unsigned char* dst;
        if (q >= n_all) {
          const int e = (q - n_all) / cpe, i = q - n_all - e * cpe;
          src = reinterpret_cast<const uint8_t*>(a.wr_next + (size_t)e * H + d0 * kUnit + 4 * i);
          dst = reinterpret_cast<unsigned char*>(wsl + e * wst + 4 * i);
        } else if (q < n_g) {
          const int u = q / (2 * ngs), rem = q - u * 2 * ngs, m = rem / ngs, i = rem - m * ngs;
          if (16 * i >= tile_n[u] * (int)L.ngh * 2) continue;  // the tile's scale rows only
          const int sq = tile_s[u], r0 = tile_r0[u];
          src = a.pool + (size_t)seg_slot[sq] * a.record_bytes + a.off_s[m] + (size_t)r0 * L.ngh * 2u + 16u * i;
          dst = smem + L.gsc + (size_t)(u * 2 + m) * L.scg + 16u * i;
        } else {
          const int q2 = q - n_g, sq = q2 / nds, i = q2 - sq * nds;
          src = a.pool + (size_t)seg_slot[sq] * a.record_bytes + a.off_s[2] + (size_t)d0 * kUnit * L.ngi * 2u + 16u * i;
          dst = smem + L.dsc + (size_t)sq * a.max_units_d * L.scd + 16u * i;
        }
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
      }
      asm volatile("cp.async.commit_group;" ::: "memory");
    }
  }

  // ------------------------------------------------ 4. gate/up + SwiGLU
  float* redg = reinterpret_cast<float*>(smem + L.redg);
  const int g = lane >> 2, cq = lane & 3;
  const bool has_tok = g == 0;
  if (warp < kD1Warps) {
    const int ngh = (int)L.ngh;
    const int gw0 = (warp * ngh) / kD1Warps, gw1 = ((warp + 1) * ngh) / kD1Warps;
    // the scale rows (this thread's copies, then every consumer's)
    asm volatile("cp.async.wait_all;" ::: "memory");
    asm volatile("bar.sync 1, %0;" ::"n"(kD1Warps * 32) : "memory");
    for (int u = 0; u < nu && gw0 < gw1; ++u) {
      if (!mbar_wait_sleep(&bars[u], par, abort_flag, a.r.err)) break;
      if (u < 4 && warp == 0) trace_mark(tr, 9 + u);
      const unsigned char* unit = gcode + (size_t)u * 2u * L.ug;
      const __half* gs = reinterpret_cast<const __half*>(smem + L.gsc + (size_t)u * 2u * L.scg);
      const __half* us = gs + L.scg / 2u;
      for (int gi = gw0; gi < gw1; ++gi) {
        float d[1][2][4];
        quad_groups_mma<2, CPG, 1>(d, unit, rowg, L.ug, gi, g, cq, xb + gi * (4 * CPG), has_tok);
        if (cq == 0) {
          const float cc = xc[gi];
          float* rp = redg + ((size_t)(u * ngh + gi) * 2) * kUnit;
          rp[g] = __half2float(gs[g * ngh + gi]) * (d[0][0][0] - cc);
          rp[kUnit + g] = __half2float(us[g * ngh + gi]) * (d[0][1][0] - cc);
          rp[g + 8] = __half2float(gs[(g + 8) * ngh + gi]) * (d[0][0][2] - cc);
          rp[kUnit + g + 8] = __half2float(us[(g + 8) * ngh + gi]) * (d[0][1][2] - cc);
        }
      }
      if (u < 4) trace_mark(tr, 13 + u);
    }
  }
  __syncthreads();
  if (!*abort_flag) {
    // h = fp16(silu(g) * u), group partials summed in group order, for the
    // tiles' valid rows
    const int ngh = (int)L.ngh;
    for (int q = tid; q < nu * kUnit; q += kD1Threads) {
      const int u = q / kUnit, row = q - u * kUnit;
      if (row >= tile_n[u]) continue;
      float gv = 0.f, uv = 0.f;
      for (int gi = 0; gi < ngh; ++gi) {
        const float* rp = redg + ((size_t)(u * ngh + gi) * 2) * kUnit;
        gv += rp[row];
        uv += rp[kUnit + row];
      }
      a.h[(size_t)tile_s[u] * I + tile_r0[u] + row] = __float2half_rn(silu_fast(gv) * uv);
    }
  }
  __syncthreads();
  trace_mark(tr, 17);
  if (tid == 0) {
    // every CTA counts itself, also after a failure, so no CTA waits in vain
    const uint32_t base = (s_base[1] - s_base[1] % (uint32_t)grid + (uint32_t)layer * (uint32_t)grid) % mod;
    epoch_arrive(gu_done, mod);
    epoch_wait(gu_done, base, mod, (uint32_t)grid, abort_flag, a.r.err);
    trace_mark(tr, 18);
  }
  __syncthreads();

  // ------------------------------------------------------------- 5. down
  // Each warp takes a run of (down unit, segment, group) tasks, four groups
  // of one segment at a time where it can. Its 32 lanes load the h words of
  // those groups straight from global memory (L2), stage them in fragment
  // order in a per-warp scratch (the consumed gate/up code rows) and reduce
  // each group's sums over the lanes holding it, so no block-wide staging
  // step sits between the count and the MMAs.
  float* redd = reinterpret_cast<float*>(smem + L.redd);
  const int ngi = (int)L.ngi;
  constexpr int WPG = 4 * CPG;  // h words per group
  if (warp < kD1Warps && ndu > 0 && !*abort_flag) {
    const int ntask = ndu * nseg * ngi;
    const int q0 = (warp * ntask) / kD1Warps, q1 = ((warp + 1) * ntask) / kD1Warps;
    uint4* scratch = reinterpret_cast<uint4*>(smem + L.hb) + (size_t)warp * 4 * WPG;
    const int nwh = I / 8;  // words of h
    int waited = -1;
    for (int q = q0; q < q1;) {
      const int du = q / (nseg * ngi), rem = q - du * nseg * ngi;
      const int sq = rem / ngi, gi = rem - sq * ngi;
      const int ng = (q + 4 <= q1 && gi + 4 <= ngi) ? 4 : 1;
      // h words of groups gi .. gi + ng - 1, word w of the block on lane w % 32
      const uint4* hsrc = reinterpret_cast<const uint4*>(a.h + (size_t)sq * I) + (size_t)gi * WPG;
      uint4 hv[(4 * WPG + 31) / 32];
      float2 hsum[(4 * WPG + 31) / 32];
#pragma unroll
      for (int i = 0; i < (4 * WPG + 31) / 32; ++i) {
        const int w = lane + 32 * i;
        hv[i] = (w < ng * WPG && gi * WPG + w < nwh) ? __ldcg(hsrc + w) : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int i = 0; i < (4 * WPG + 31) / 32; ++i) {
        const int w = lane + 32 * i;
        hsum[i] = word_sums(hv[i]);
        if (w < 4 * WPG) scratch[w] = b_frag(hv[i]);
        // butterfly over the WPG lanes that hold this group's words
#pragma unroll
        for (int o = WPG / 2; o > 0; o >>= 1) {
          hsum[i].x += __shfl_xor_sync(0xffffffffu, hsum[i].x, o);
          hsum[i].y += __shfl_xor_sync(0xffffffffu, hsum[i].y, o);
        }
      }
      float cc[4];
#pragma unroll
      for (int n = 0; n < 4; ++n) {
        const int w = n * WPG;  // first word of group n: lane w % 32, register w / 32
        float v = 0.f;
#pragma unroll
        for (int i = 0; i < (4 * WPG + 31) / 32; ++i) {
          const float x = __shfl_sync(0xffffffffu, 1032.f * hsum[i].x + 72.f * hsum[i].y, w & 31);
          if (i == w / 32) v = x;
        }
        cc[n] = v;
      }
      __syncwarp();
      if (sq != waited) {
        if (!mbar_wait_sleep(&bars[mug + sq], par, abort_flag, a.r.err)) break;
        if (waited < 0 && warp == 0) trace_mark(tr, 19);
        if (waited < 0) trace_mark(trw, 21);
        waited = sq;
      }
      const unsigned char* unit = dcode + (size_t)sq * L.ud + (size_t)du * kUnit * rowd;
      const __half* ds = reinterpret_cast<const __half*>(smem + L.dsc + ((size_t)sq * a.max_units_d + du) * L.scd);
      float* rp0 = redd + ((size_t)(du * ns_max + sq) * ngi) * kUnit;
      if (ng == 4) {
        float d[4][1][4];
        quad_groups_mma<1, CPG, 4>(d, unit, rowd, 0u, gi, g, cq, scratch, has_tok);
        if (cq == 0)
#pragma unroll
          for (int n = 0; n < 4; ++n) {
            float* rp = rp0 + (size_t)(gi + n) * kUnit;
            rp[g] = __half2float(ds[g * ngi + gi + n]) * (d[n][0][0] - cc[n]);
            rp[g + 8] = __half2float(ds[(g + 8) * ngi + gi + n]) * (d[n][0][2] - cc[n]);
          }
      } else {
        float d[1][1][4];
        quad_groups_mma<1, CPG, 1>(d, unit, rowd, 0u, gi, g, cq, scratch, has_tok);
        if (cq == 0) {
          float* rp = rp0 + (size_t)gi * kUnit;
          rp[g] = __half2float(ds[g * ngi + gi]) * (d[0][0][0] - cc[0]);
          rp[g + 8] = __half2float(ds[(g + 8) * ngi + gi]) * (d[0][0][2] - cc[0]);
        }
      }
      __syncwarp();  // the scratch is rewritten by the next block
      q += ng;
    }
    trace_mark(tr, 20);
    trace_mark(trw, 22);
  }
  __syncthreads();
  trace_mark(tr, 23);
  float* y = reinterpret_cast<float*>(smem + L.y);
  const int ydim = a.max_units_d * kUnit;  // y rows per segment
  if (!*abort_flag)
    for (int q = tid; q < nseg * ndr; q += kD1Threads) {
      // y_s[row]: the segment's group partials summed in group order
      const int sq = q / ndr, lr = q - sq * ndr;
      const int du = lr / kUnit, row = lr - du * kUnit;
      const float* rp = redd + ((size_t)(du * ns_max + sq) * ngi) * kUnit + row;
      float v = 0.f;
      for (int gi = 0; gi < ngi; ++gi) v += rp[gi * kUnit];
      y[sq * ydim + lr] = v;
    }
  __syncthreads();
  if (!*abort_flag) {
    // out[row] = sum_j w_j y_j[row] in rank order, then the shared expert;
    // one FP16 rounding; the residual
    for (int lr = tid; lr < ndr; lr += kD1Threads) {
      float acc = 0.f;
      for (int j = 0; j < k; ++j) acc = fmaf(sel_w[j], y[pos_of_rank[j] * ydim + lr], acc);
      if (a.r.has_shared) acc += y[k * ydim + lr];
      __half o = __float2half_rn(acc);
      const int orow = d0 * kUnit + lr;
      if (a.x_res) o = __float2half_rn(__half2float(__ldcg(a.x_res + orow)) + __half2float(o));
      a.out[orow] = o;
      if (STACK) xo[lr] = __half2float(o);
    }
  }
  trace_mark(tr, 24);
  if (bid == 0 && warp == kD1Producer && !*abort_flag) {
    // publish the routing (moe_layer_routing, the user's ids / weights):
    // only read after the launch, so off the critical path
    if (lane < k) {
      const int id = sel_id[lane], pr = pos_of_rank[lane];
      const float wv = sel_w[lane];
      a.r.ids[lane] = id;
      a.r.w[lane] = wv;
      if (a.r.ids_user) a.r.ids_user[lane] = id;
      if (a.r.w_user) a.r.w_user[lane] = wv;
      a.r.perm[pr] = lane;
      a.r.inv_perm[lane] = pr;
    }
    for (int e = lane; e <= E; e += 32) {
      int below = 0, hit = 0;
      for (int j = 0; j < k; ++j) {
        below += sel_id[j] < e ? 1 : 0;
        hit += sel_id[j] == e ? 1 : 0;
      }
      a.r.offsets[e] = below;
      if (e < E) a.r.counts[e] = hit;
    }
    if (lane < nseg) {
      a.r.seg_expert[lane] = seg_expert[lane];
      a.r.seg_start[lane] = lane;
      a.r.seg_count[lane] = 1;
    }
    if (lane == 0) *a.r.num_seg = nseg;
  }
  if constexpr (STACK) {
    if (a.wr_next) {
      // the next layer's partial logits over these rows; the count releases
      // them and the rows of the output (the next layer's input)
      __syncthreads();
      if (!*abort_flag) d1_row_partials(xo, wsl, wst, E, ndr, a.part_out + (size_t)bid * E);
      __syncthreads();
      if (tid == 0) epoch_arrive(logits_ready, mod);
    }
  }

  // ---------------------------------------------------------- teardown
  if (tid == 0 && *abort_flag && *issued) {
    // let every issued copy land before the CTA's shared memory is released
    for (int u = 0; u < nu; ++u) mbar_wait(&bars[u], par, nullptr, nullptr);
    for (int sq = 0; sq < ns_max; ++sq) mbar_wait(&bars[mug + sq], par, nullptr, nullptr);
  }
  trace_mark(tr, 25);
  if (STACK) __syncthreads();  // the next layer reuses the shared memory
}

template <int NV, int CPG>
__global__ void __launch_bounds__(kD1Threads, 1) k_decode1(const __grid_constant__ Decode1Args a) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  const D1Layout L = d1_layout(a);
  unsigned char* smem = smem_raw + (((smem_u32(smem_raw) + 1023u) & ~1023u) - smem_u32(smem_raw));
  if (threadIdx.x == 0) *reinterpret_cast<volatile int*>(smem + L.ctl) = 0;  // abort flag
  d1_layer<NV, CPG, false>(a, smem, L, 0, true);
}

// The layers of a stack in one launch: layer l + 1 starts when every CTA has
// written its rows of layer l's output and its partial logits of layer l + 1
// (one grid-wide count per layer boundary instead of a launch). A CTA that
// gave up in one layer skips the work of the later ones but still counts
// itself at every step.
template <int NV, int CPG>
__global__ void __launch_bounds__(kD1Threads, 1) k_decode1_stack(const __grid_constant__ Decode1Stack S) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  const D1Layout L = d1_layout(S.layer[0]);
  unsigned char* smem = smem_raw + (((smem_u32(smem_raw) + 1023u) & ~1023u) - smem_u32(smem_raw));
  if (threadIdx.x == 0) *reinterpret_cast<volatile int*>(smem + L.ctl) = 0;  // abort flag
  for (int l = 0; l < S.n_layers; ++l) d1_layer<NV, CPG, true>(S.layer[l], smem, L, l, l == S.trace_layer);
}

template <int NV, int CPG>
cudaError_t launch_decode1_t(const Decode1Args& a, int grid, cudaStream_t s, bool pdl) {
  const size_t smem = decode1_smem_bytes(a);
  if (smem == 0) return cudaErrorInvalidValue;
  cudaError_t e = ensure_smem(k_decode1<NV, CPG>, smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kD1Threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, k_decode1<NV, CPG>, a);
}

template <int NV>
cudaError_t launch_decode1_nv(const Decode1Args& a, int grid, cudaStream_t s, bool pdl) {
  return a.G == 64 ? launch_decode1_t<NV, 2>(a, grid, s, pdl) : launch_decode1_t<NV, 4>(a, grid, s, pdl);
}

template <int NV, int CPG>
cudaError_t launch_decode1_stack_t(const Decode1Stack& st, int grid, cudaStream_t s, bool pdl) {
  const size_t smem = decode1_smem_bytes(st.layer[0]);
  if (smem == 0) return cudaErrorInvalidValue;
  cudaError_t e = ensure_smem(k_decode1_stack<NV, CPG>, smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kD1Threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, k_decode1_stack<NV, CPG>, st);
}

template <int NV>
cudaError_t launch_decode1_stack_nv(const Decode1Stack& st, int grid, cudaStream_t s, bool pdl) {
  return st.layer[0].G == 64 ? launch_decode1_stack_t<NV, 2>(st, grid, s, pdl)
                             : launch_decode1_stack_t<NV, 4>(st, grid, s, pdl);
}

}  // namespace

int decode1_max_tiles(int nseg, int I, int grid) {
  const int gpe = I / 8;
  int mx = 0;
  for (int b = 0; b < grid; ++b) {
    const int g0 = (int)((long long)b * nseg * gpe / grid), g1 = (int)((long long)(b + 1) * nseg * gpe / grid);
    int ds0, ds1, ds2;
    const int n = walk_tiles(g0, g1, gpe, -1, &ds0, &ds1, &ds2);
    mx = n > mx ? n : mx;
  }
  return mx;
}

size_t decode1_smem_bytes(const Decode1Args& a) {
  if (a.r.H % kUnit || a.I % kUnit || (a.G != 64 && a.G != 128)) return 0;
  const D1Layout L = d1_layout(a);
  return L.total <= kSmemBudget ? L.total : 0;
}

cudaError_t launch_decode1_stack(const Decode1Stack& st, int grid, cudaStream_t s, bool pdl) {
  if (st.n_layers < 1 || st.n_layers > kD1MaxLayers || grid > kD1Runs * kD1RunMax) return cudaErrorInvalidValue;
  const Decode1Args& a = st.layer[0];
  for (int l = 0; l < st.n_layers; ++l) {
    const Decode1Args& b = st.layer[l];
    // one shape for every layer (one layout, one template), one counter pair
    if (!b.stack || b.r.T != 1 || b.r.H != a.r.H || b.I != a.I || b.r.E != a.r.E || b.r.k != a.r.k || b.G != a.G ||
        b.r.has_shared != a.r.has_shared || b.ctr != a.ctr || b.ctr_mod != a.ctr_mod || !b.part_in || !b.part_out ||
        (l + 1 < st.n_layers) != (b.wr_next != nullptr))
      return cudaErrorInvalidValue;
  }
  if (a.ctr_mod == 0 || a.ctr_mod % (uint32_t)grid) return cudaErrorInvalidValue;
  if (a.r.E <= 64) return launch_decode1_stack_nv<2>(st, grid, s, pdl);
  if (a.r.E <= 128) return launch_decode1_stack_nv<4>(st, grid, s, pdl);
  return cudaErrorInvalidValue;  // the partial logits of larger E: per-layer launches
}

cudaError_t launch_decode1(const Decode1Args& a, int grid, cudaStream_t s, bool pdl) {
  if (a.stack) return cudaErrorInvalidValue;
  if (a.r.T != 1 || a.ctr_mod == 0 || a.ctr_mod % (uint32_t)grid) return cudaErrorInvalidValue;
  if (a.r.E <= 64) return launch_decode1_nv<2>(a, grid, s, pdl);
  if (a.r.E <= 128) return launch_decode1_nv<4>(a, grid, s, pdl);
  if (a.r.E <= 256) return launch_decode1_nv<8>(a, grid, s, pdl);
  if (a.r.E <= 512) return launch_decode1_nv<16>(a, grid, s, pdl);
  return launch_decode1_nv<32>(a, grid, s, pdl);
}

}  // namespace moe
