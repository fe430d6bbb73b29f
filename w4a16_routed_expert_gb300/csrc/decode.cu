// Decode megakernel: the whole layer forward for a small batch (T <= 16,
// fully resident table) in one cooperative launch, one CTA per SM.
//
// The multi-kernel path pays a launch boundary and a pipeline ramp between
// routing, gate/up, down and the combine; at batch 1 each of those costs as
// much as streaming the weights. Here, inside one persistent grid whose CTAs
// are all resident (cooperative launch):
//   1. router logits: (expert, part) partial dot products spread over every
//      warp of the grid;
//   2. a grid-wide arrival count on the partials; then every CTA sums them
//      in order and computes the top-k, the permutation and the segment list
//      itself, into its own shared memory (identical results in every CTA,
//      no second grid hop); CTA 0 also publishes them to global memory;
//   3. gate/up + SwiGLU work items on the tensor cores (tcgemv_dev.cuh:
//      codes dequantised in registers into mma.sync fragments);
//   4. down work items, whose weights the producer streams into the ring
//      while gate/up items are still being computed; the consumers wait once
//      per segment for that segment's gate/up counter before reading h;
//   5. every down item counts on a per-row-block counter; the CTA that
//      completes a row block performs the weighted combine for those rows
//      (fixed order: ranks j = 0..k-1, then the shared expert).
// Warp roles: 16 consumer warps compute items out of a shared-memory ring and
// hand their K-part partial sums over in shared memory; one producer warp
// fills the ring with TMA copies; one finisher warp reduces the partials,
// writes h or y, turns each finished item into its GPU-scope counter update
// and runs the combines, so no consumer waits on an epilogue, a release or
// an atomic.
// Every cross-CTA wait is a bounded spin; on time-out the CTA records an
// error, stops, lets its issued copies land and still passes the final
// ticket, whose last holder resets all counters for the next launch.
#include <mutex>

#include "route_dev.cuh"
#include "tcgemv_dev.cuh"

namespace moe {

namespace {

constexpr int kProducerWarp = kTcWarps;
constexpr int kSignalWarp = kTcWarps + 1;
constexpr int kDecodeThreads = (kTcWarps + 2) * 32;

struct DecodeHdr {
  uint64_t full[kDecodeMaxStages];   // producer -> consumers: the item's bytes landed
  uint64_t empty[kDecodeMaxStages];  // consumers -> producer: the stage is free
  TcRedBars red;                     // consumers <-> finisher: K-part partials
  int ncombine;                      // row blocks listed for the CTA-wide combine
  int abort_flag;
  int issued;
  int last;
};
static_assert(sizeof(DecodeHdr) <= kHdrBytes, "decode header exceeds its reserved bytes");

// Weighted combine of down row block rbi by one warp (the signalling warp of
// the CTA that completed it): out[t][row] = sum_j w[t][j] * y[(t, j)][row]
// in rank order, then the shared expert, the FP16 rounding and the residual.
// The same arithmetic, in the same order, as the multi-kernel combine.
__device__ __noinline__ void decode_combine_rows(const DecodeArgs& a, const TcGemvArgs& d, int rbi,
                                                    const float* s_w, int lane) {
  const int T = a.r.T, H = a.r.H, k = a.r.k, Tk = T * k;
  const int r0 = rbi * d.rb;
  const int nrows = min(d.rb, H - r0);
#pragma unroll 2
  for (int q = lane; q < nrows * T; q += 32) {
    const int t = q / nrows, row = r0 + q % nrows;
    const float* yp = d.y_out + (size_t)t * k * H + row;
    float acc = 0.f;
    int j = 0;
    for (; j + 8 <= k; j += 8) {
      float v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) v[u] = __ldcg(yp + (size_t)(j + u) * H);
#pragma unroll
      for (int u = 0; u < 8; ++u) acc = fmaf(s_w[t * k + j + u], v[u], acc);
    }
    for (; j < k; ++j) acc = fmaf(s_w[t * k + j], __ldcg(yp + (size_t)j * H), acc);
    if (a.has_shared) acc += __ldcg(d.y_out + (size_t)(Tk + t) * H + row);
    __half o = __float2half_rn(acc);
    if (a.x_res) o = __float2half_rn(__half2float(a.x_res[(size_t)t * H + row]) + __half2float(o));
    a.out[(size_t)t * H + row] = o;
  }
}

// Dynamic shared memory: header, then (1024-byte aligned) the ring, the B
// fragments, the group constants, the K-part partials (two buffers) and the
// routing arrays.
struct DecodeSmem {
  uint32_t ring, bs, cs, red, route, total;
};
__host__ __device__ inline DecodeSmem decode_smem_layout(const DecodeArgs& a, int stages) {
  DecodeSmem L;
  const uint32_t Tk = (uint32_t)(a.r.T * a.r.k), E = (uint32_t)a.r.E, ns = (uint32_t)a.ns;
  L.ring = kHdrBytes;  // rounded up to 1024 in the kernel (slack below)
  L.bs = L.ring + 1024u + (uint32_t)stages * a.slot_bytes;
  L.cs = L.bs + (uint32_t)a.bs_chunks * ns * 64u;
  L.red = L.cs + (((uint32_t)a.cs_groups * ns * 4u + 15u) & ~15u);
  L.route = L.red + ((2u * (uint32_t)tc_red_words((int)ns) * 4u + 15u) & ~15u);
  // (+3: alignment of the finish scratch)
  L.total = L.route + (4u * Tk + 5u * E + 11u + (uint32_t)route_finish_scratch_ints(a.r.T, a.r.E, a.r.k)) * 4u;
  return L;
}

// NV: router values per lane (E <= 32 NV); TMAX: the largest T of the
// launch (1, 4 or 16), so that only the loops and routing paths a batch of
// that size needs are compiled into the instance it runs.
template <int NV, int TMAX>
__global__ void __launch_bounds__(kDecodeThreads, 1) k_decode(const __grid_constant__ DecodeArgs a) {
  extern __shared__ __align__(128) unsigned char smem[];
  DecodeHdr* hdr = reinterpret_cast<DecodeHdr*>(smem);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int S = a.stages;
  const int T = a.r.T, E = a.r.E, k = a.r.k;
  const int Tk = T * k;
  const int NS = a.ns;
  uint32_t* logits_done = a.ctr;
  uint32_t* final_ticket = a.ctr + 1;
  uint32_t* done_gu = a.ctr + 2;
  uint32_t* done_dn = a.ctr + 2 + (E + 1);

  const DecodeSmem lay = decode_smem_layout(a, S);
  const uint32_t sbase = smem_u32(smem);
  unsigned char* ring = smem + (((sbase + lay.ring + 1023u) & ~1023u) - sbase);
  uint4* Bs = reinterpret_cast<uint4*>(smem + lay.bs);
  float* Cs = reinterpret_cast<float*>(smem + lay.cs);
  float* red = reinterpret_cast<float*>(smem + lay.red);
  // routing results of this CTA, sized for this E and T*k
  int32_t* s_ids = reinterpret_cast<int32_t*>(smem + lay.route);  // [Tk]
  float* s_w = reinterpret_cast<float*>(s_ids + Tk);               // [Tk]
  int32_t* s_counts = reinterpret_cast<int32_t*>(s_w + Tk);        // [E]
  int32_t* s_off = s_counts + E;                                   // [E+1]
  int32_t* s_perm = s_off + E + 1;                                 // [Tk]
  int32_t* s_inv = s_perm + Tk;                                    // [Tk]
  int32_t* s_sexp = s_inv + Tk;                                    // [E+1]
  int32_t* s_sstart = s_sexp + E + 1;                              // [E+1]
  int32_t* s_scount = s_sstart + E + 1;                            // [E+1]
  int32_t* s_nseg = s_scount + E + 1;                              // [1] (+3 pad)
  // route_finish_scratch_ints(T, E, k), 16-byte aligned
  int32_t* s_scratch = s_nseg + 4 + ((4u - ((smem_u32(s_nseg + 4) >> 2) & 3u)) & 3u);

  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&hdr->full[s], 1);
      mbar_init(&hdr->empty[s], kTcWarps);
    }
    tc_red_bars_init(&hdr->red);
    hdr->abort_flag = 0;
    hdr->issued = 0;
    hdr->last = 0;
    hdr->ncombine = 0;
    fence_mbar_init();
  }
  if (warp == kProducerWarp && lane == 0) {
    prefetch_tmap(&a.tm_gate);
    prefetch_tmap(&a.tm_up);
    prefetch_tmap(&a.tm_down);
  }
  // Launched with programmatic stream serialisation (when available): the
  // next kernel may begin launching now, and nothing above touched global
  // memory; wait here until the previous kernel has completed and its
  // writes (the input tokens, this layer's counters) are visible.
  pdl_trigger();
  pdl_wait();
  __syncthreads();
  volatile int* abort_flag = &hdr->abort_flag;
  unsigned long long* tr = (tid == 0) ? a.trace : nullptr;
  trace_mark(tr, 0);

  // ------------------------------------------------ 1. router logits (FP32)
  // (expert, part) tasks spread over every warp of the grid; the partials are
  // summed in order when the logits are read (routing below).
  {
    const int nw = gridDim.x * (kDecodeThreads / 32);
    for (int q = warp * gridDim.x + blockIdx.x; q < E * kLogitParts; q += nw)
      warp_logit_partial<TMAX>(a.r, q / kLogitParts, q % kLogitParts, a.r.logit_part);
  }
  __syncthreads();
  trace_mark(tr, 1);
  if (tid == 0) {
    // bar.sync above orders every warp's partials before this release
    red_release_add(logits_done, 1u);
    wait_count(logits_done, gridDim.x, abort_flag, a.r.err);
  }
  __syncthreads();
  trace_mark(tr, 2);

  int nseg = 0;
  if (!*abort_flag) {
    // -------------------------- 2. routing into this CTA's shared memory
    RouteArgs L = a.r;
    L.ids = s_ids;
    L.w = s_w;
    L.ids_user = blockIdx.x == 0 ? a.r.ids_user : nullptr;
    L.w_user = blockIdx.x == 0 ? a.r.w_user : nullptr;
    L.counts = s_counts;
    L.offsets = s_off;
    L.perm = s_perm;
    L.inv_perm = s_inv;
    L.seg_expert = s_sexp;
    L.seg_start = s_sstart;
    L.seg_count = s_scount;
    L.num_seg = s_nseg;
    route_finish_cta<NV, TMAX == 1>(L, s_scratch, a.r.logit_part, tr);
    __syncthreads();
    trace_mark(tr, 4);
    nseg = *s_nseg;
    if (blockIdx.x == 0) {
      // publish for moe_layer_routing and the routing outputs
      for (int i = tid; i < Tk; i += blockDim.x) {
        a.r.ids[i] = s_ids[i];
        a.r.w[i] = s_w[i];
        a.r.perm[i] = s_perm[i];
        a.r.inv_perm[i] = s_inv[i];
      }
      for (int i = tid; i < E; i += blockDim.x) a.r.counts[i] = s_counts[i];
      for (int i = tid; i <= E; i += blockDim.x) a.r.offsets[i] = s_off[i];
      if (tid == 0) *a.r.num_seg = nseg;
    }
  }

  // ------------------------------------ 3./4. gate/up then down work items
  TcGemvArgs g = a.g, d = a.d;
  g.seg_expert = d.seg_expert = s_sexp;
  g.seg_start = d.seg_start = s_sstart;
  g.seg_count = d.seg_count = s_scount;
  g.perm = d.perm = s_perm;
  const int nrb_g = (g.N + g.rb - 1) / g.rb;
  const int nrb_d = (d.N + d.rb - 1) / d.rb;
  const int tot_g = nseg * nrb_g, tot_d = nseg * nrb_d;
  // balanced contiguous split: CTA b takes items [b * tot / grid, (b+1) * tot / grid)
  const int fg = (int)((long long)blockIdx.x * tot_g / gridDim.x);
  const int fd = (int)((long long)blockIdx.x * tot_d / gridDim.x);
  const int ng_it = (int)((long long)(blockIdx.x + 1) * tot_g / gridDim.x) - fg;
  const int nd_it = (int)((long long)(blockIdx.x + 1) * tot_d / gridDim.x) - fd;
  const int n_it = *abort_flag ? 0 : ng_it + nd_it;
  const int combine_cap = route_finish_scratch_ints(T, E, k);  // the routing scratch, free after routing
  const uint32_t gu_target = (uint32_t)nrb_g;  // gate/up items per segment
  const uint32_t dn_target = (uint32_t)nseg;   // down items per row block

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t pol = l2_policy_evict_first();
      for (int it = 0; it < n_it; ++it) {
        const int st = it % S;
        const uint32_t ph = (uint32_t)(it / S) & 1u;
        if (!mbar_wait(&hdr->empty[st], ph ^ 1u, abort_flag, a.r.err)) break;
        unsigned char* slot = ring + (size_t)st * a.slot_bytes;
        if (it < ng_it)
          tc_issue_item<true>(g, &a.tm_gate, &a.tm_up, fg + it, nrb_g, slot, &hdr->full[st], pol);
        else
          tc_issue_item<false>(d, &a.tm_down, &a.tm_down, fd + it - ng_it, nrb_d, slot, &hdr->full[st], pol);
        hdr->issued = it + 1;
      }
    }
  } else if (warp == kSignalWarp) {
    // ----------------------------------------------------------- finisher
    // Token tile by token tile (the consumers' order): wait for the K-part
    // partials, write the outputs (h with SwiGLU, or y), free the buffer.
    // Gate/up items add to their segment's counter, one release per run of
    // this CTA's items of a segment; down items count on their row block
    // once all of this CTA's down outputs are written, and the item that
    // completes a row block leads to that block's combine. Every output this
    // warp writes precedes its own GPU-scope release.
    uint32_t pending = 0;
    int ti = 0;
    bool ok = true;
    for (int it = 0; it < n_it && ok; ++it) {
      const bool gu = it < ng_it;
      const int item = gu ? fg + it : fd + it - ng_it;
      const int nrb = gu ? nrb_g : nrb_d;
      const int sgi = item / nrb, rbi = item - sgi * nrb;
      const int cnt = s_scount[sgi];
      for (int tb = 0; tb < cnt; tb += kTcMaxTok) {
        const int ntok = min(kTcMaxTok, cnt - tb);
        const int b = ti & 1;
        int w = 1;
        if (lane == 0) w = mbar_wait(&hdr->red.full[b], (uint32_t)(ti >> 1) & 1u, abort_flag, a.r.err);
        w = __shfl_sync(0xffffffffu, w, 0);
        if (!w) {
          ok = false;
          break;
        }
        const float* rbuf = red + b * tc_red_words(NS);
        if (gu)
          tc_finish_warp<true>(g, sgi, rbi, tb, ntok, NS, rbuf, lane);
        else
          tc_finish_warp<false>(d, sgi, rbi, tb, ntok, NS, rbuf, lane);
        __syncwarp();
        if (lane == 0) mbar_arrive(&hdr->red.free_[b]);
        ++ti;
      }
      if (!ok) break;
      if (gu) {
        // one release per run of this CTA's items of a segment
        ++pending;
        const int nx = it + 1;
        if (nx >= ng_it || (fg + nx) / nrb_g != sgi) {
          __syncwarp();
          if (lane == 0) red_release_add(done_gu + sgi, pending);
          pending = 0;
        }
      }
    }
    // down items: every y of this CTA written above; then one row-block count
    // per item, lane i for item i, all in flight together. The row blocks
    // this CTA completes are listed for the whole CTA to combine after the
    // teardown barrier (or combined here if the list would overflow).
    __syncwarp();
    int nlist = 0;
    for (int i0 = 0; ok && i0 < nd_it; i0 += 32) {
      const int i = i0 + lane;
      int last = 0;
      if (i < nd_it) {
        const int rbi = (fd + i) % nrb_d;
        last = (atom_acq_rel_add(done_dn + rbi, 1u) + 1u == dn_target) ? 1 : 0;
      }
      uint32_t mask = __ballot_sync(0xffffffffu, last);
      __syncwarp();
      // each lane's acq_rel increment observed every other CTA's release
      while (mask) {
        const int l = __ffs(mask) - 1;
        mask &= mask - 1;
        const int rbi = (fd + i0 + l) % nrb_d;
        if (nlist < combine_cap) {
          if (lane == 0) s_scratch[nlist] = rbi;
          ++nlist;
        } else {
          decode_combine_rows(a, d, rbi, s_w, lane);
        }
      }
    }
    if (lane == 0) hdr->ncombine = nlist;
    if (lane == 0 && a.trace) {
      unsigned long long t;
      asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
      a.trace[blockIdx.x * kTraceStamps + 9] = t;
    }
  } else {
    // ----------------------------------------------------------- consumers
    // Every consumer warp runs the same sequence of named barriers (it
    // depends only on the routing in shared memory), also after a failed
    // wait: the work is then skipped in effect (stale data), never the
    // barrier, so no warp can be left waiting. Barriers are only needed when
    // the B fragments are rebuilt; otherwise the warps run independently,
    // handing their partials to the finisher through the two buffers.
    int b_seg = -1, b_tb = -1, b_gu = -1;  // token tile the B buffer holds
    int ready_seg = -1;
    int ti = 0;
    if (n_it > 0 && ng_it > 0) {
      // the first item's token fragments while its codes are still in flight
      const int sgi0 = fg / nrb_g;
      tc_build_b<false>(g, sgi0, 0, min(kTcMaxTok, s_scount[sgi0]), NS, Bs, Cs, tid);
      b_seg = sgi0;
      b_tb = 0;
      b_gu = 1;
      tc_bar();
    }
    for (int it = 0; it < n_it; ++it) {
      const int st = it % S;
      const uint32_t ph = (uint32_t)(it / S) & 1u;
      mbar_wait(&hdr->full[st], ph, abort_flag, a.r.err);
      if (it < kTraceItems) trace_mark(tr, kTracePhases + 2 * it);
      const unsigned char* slot = ring + (size_t)st * a.slot_bytes;
      const bool gu = it < ng_it;
      const int item = gu ? fg + it : fd + it - ng_it;
      const int nrb = gu ? nrb_g : nrb_d;
      const int sgi = item / nrb;
      const int cnt = s_scount[sgi];
      if (it == 0) trace_mark(tr, 5);
      for (int tb = 0; tb < cnt; tb += kTcMaxTok) {
        const int ntok = min(kTcMaxTok, cnt - tb);
        if (sgi != b_seg || tb != b_tb || (int)gu != b_gu) {
          tc_bar();  // every consumer warp is done with the previous B fragments
          if (gu) {
            tc_build_b<false>(g, sgi, tb, ntok, NS, Bs, Cs, tid);
          } else {
            const bool first_dn = ready_seg < 0;
            if (first_dn) trace_mark(tr, 12);
            if (sgi != ready_seg) {
              // h of this segment: every gate/up item of it, from every CTA
              int w = 1;
              if (lane == 0) w = wait_count(done_gu + sgi, gu_target, abort_flag, a.r.err);
              w = __shfl_sync(0xffffffffu, w, 0);
              __syncwarp();
              (void)w;  // on failure the abort flag is set; the barriers still run
              ready_seg = sgi;
            }
            if (first_dn) trace_mark(tr, 13);
            tc_build_b<true>(d, sgi, tb, ntok, NS, Bs, Cs, tid);
            if (first_dn) trace_mark(tr, 14);
          }
          b_seg = sgi;
          b_tb = tb;
          b_gu = gu;
          tc_bar();
        }
        const int b = ti & 1;
        // the finisher has read this buffer (token tile ti - 2)
        if (lane == 0) mbar_wait(&hdr->red.free_[b], ((uint32_t)(ti >> 1) & 1u) ^ 1u, abort_flag, a.r.err);
        __syncwarp();
        float* rbuf = red + b * tc_red_words(NS);
        if (gu) {
          tc_compute<true>(g, slot, Bs, Cs, ntok, NS, rbuf, warp, lane);
        } else {
          if (it == ng_it && tb == 0) trace_mark(tr, 7);
          tc_compute<false>(d, slot, Bs, Cs, ntok, NS, rbuf, warp, lane);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&hdr->red.full[b]);
        ++ti;
      }
      if (gu && it == ng_it - 1) trace_mark(tr, 6);
      __syncwarp();
      if (lane == 0) mbar_arrive(&hdr->empty[st]);  // the slot's bytes are no longer read
      if (it < kTraceItems) trace_mark(tr, kTracePhases + 2 * it + 1);
    }
    trace_mark(tr, 8);
  }

  // ---------------------------------------------------------------- teardown
  __syncthreads();
  trace_mark(tr, 10);
  {
    // combine of the row blocks this CTA completed, every thread of the CTA:
    // out[t][row] = sum_j w[t][j] * y[(t, j)][row], then the shared expert,
    // the FP16 rounding and the residual (as decode_combine_rows)
    const int nl = hdr->ncombine;
    const int H = a.r.H;
    for (int q = tid; q < nl * d.rb * T; q += blockDim.x) {
      const int li = q / (d.rb * T), rem = q - li * (d.rb * T);
      const int t = rem / d.rb, row = s_scratch[li] * d.rb + rem % d.rb;
      if (row >= H) continue;
      const float* yp = d.y_out + (size_t)t * k * H + row;
      float acc = 0.f;
      int j = 0;
      for (; j + 8 <= k; j += 8) {
        float v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) v[u] = __ldcg(yp + (size_t)(j + u) * H);
#pragma unroll
        for (int u = 0; u < 8; ++u) acc = fmaf(s_w[t * k + j + u], v[u], acc);
      }
      for (; j < k; ++j) acc = fmaf(s_w[t * k + j], __ldcg(yp + (size_t)j * H), acc);
      if (a.has_shared) acc += __ldcg(d.y_out + (size_t)(Tk + t) * H + row);
      __half o = __float2half_rn(acc);
      if (a.x_res) o = __float2half_rn(__half2float(a.x_res[(size_t)t * H + row]) + __half2float(o));
      a.out[(size_t)t * H + row] = o;
    }
  }
  if (tid == 0 && hdr->abort_flag) {
    const int issued = hdr->issued;
    for (int s = 0; s < S && s < issued; ++s) {
      const int n = (issued - 1 - s) / S;
      mbar_wait(&hdr->full[s], (uint32_t)n & 1u, nullptr, nullptr);
    }
  }
  if (tid == 0) {
    hdr->last = (atom_acq_rel_add(final_ticket, 1u) == gridDim.x - 1) ? 1 : 0;
    trace_mark(tr, 11);
  }
  __syncthreads();
  if (hdr->last) {
    // every CTA has finished: reset the counters for the next launch
    for (int i = tid; i <= E; i += blockDim.x) done_gu[i] = 0u;
    for (int i = tid; i < nrb_d; i += blockDim.x) done_dn[i] = 0u;
    if (tid == 0) {
      *logits_done = 0u;
      *final_ticket = 0u;
    }
  }
}

template <int NV, int TMAX>
cudaError_t launch_decode_t(const DecodeArgs& a, int grid, cudaStream_t s, bool pdl) {
  const size_t smem = decode_smem_bytes(a, a.stages);
  cudaError_t e = ensure_smem(k_decode<NV, TMAX>, smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kDecodeThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, k_decode<NV, TMAX>, a);
}

template <int NV>
cudaError_t launch_decode_nv(const DecodeArgs& a, int grid, cudaStream_t s, bool pdl) {
  if (a.r.T <= 1) return launch_decode_t<NV, 1>(a, grid, s, pdl);
  if (a.r.T <= 4) return launch_decode_t<NV, 4>(a, grid, s, pdl);
  return launch_decode_t<NV, kSmallRouteMaxT>(a, grid, s, pdl);
}

// Whether a cooperative launch also accepts programmatic stream
// serialisation on this device: probed once per process with an empty
// cooperative kernel on a private stream (never inside a stream capture).
__global__ void k_coop_pdl_probe() {
  pdl_trigger();
  pdl_wait();
}
bool coop_pdl_probe_once() {
  static int state = -1;  // -1 unknown, 0 no, 1 yes
  static std::mutex mu;
  std::lock_guard<std::mutex> lock(mu);
  if (state >= 0) return state == 1;
  state = 0;
  cudaStream_t st = nullptr;
  if (cudaStreamCreateWithFlags(&st, cudaStreamNonBlocking) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2);
  cfg.blockDim = dim3(32);
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  cudaError_t e = cudaLaunchKernelEx(&cfg, k_coop_pdl_probe);
  if (e == cudaSuccess) e = cudaLaunchKernelEx(&cfg, k_coop_pdl_probe);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e == cudaSuccess) state = 1;
  cudaGetLastError();
  cudaStreamDestroy(st);
  return state == 1;
}

}  // namespace

size_t decode_smem_bytes(const DecodeArgs& a, int stages) { return decode_smem_layout(a, stages).total; }

TcGemvPlan plan_tcgemv(int N, int K, int G, bool dual, int item_bytes, bool zp) {
  TcGemvPlan p;
  const int mats = dual ? 2 : 1;
  p.rb = 16;
  while (p.rb * 2 <= N && p.rb * 2 / 16 <= kTcMaxRowTiles && mats * (p.rb * 2) * (K / 2) <= item_bytes) p.rb *= 2;
  p.rt = p.rb / 16;
  p.kparts = kTcWarps / p.rt;
  p.lkparts = 0;
  while ((1 << p.lkparts) < p.kparts) ++p.lkparts;
  p.nbox = (K / 2 + 127) / 128;
  p.code_mat_bytes = (uint32_t)p.nbox * 128u * (uint32_t)p.rb;
  const int ng = (K + G - 1) / G;
  p.sstride = ((uint32_t)p.rb * ng * 2u + 15u) & ~15u;
  p.zstride = zp ? (((uint32_t)p.rb * ng + 15u) & ~15u) : 0u;
  p.slot_bytes = ((uint32_t)mats * (p.code_mat_bytes + p.sstride + p.zstride) + 1023u) & ~1023u;
  return p;
}

bool decode_pdl_supported() { return coop_pdl_probe_once(); }

cudaError_t launch_decode(const DecodeArgs& a, int grid, cudaStream_t s, bool pdl) {
  if (a.r.T < 1 || a.r.T > kSmallRouteMaxT) return cudaErrorInvalidValue;
  if (a.r.E <= 64) return launch_decode_nv<2>(a, grid, s, pdl);
  if (a.r.E <= 128) return launch_decode_nv<4>(a, grid, s, pdl);
  if (a.r.E <= 256) return launch_decode_nv<8>(a, grid, s, pdl);
  if (a.r.E <= 512) return launch_decode_nv<16>(a, grid, s, pdl);
  return launch_decode_nv<32>(a, grid, s, pdl);
}

}  // namespace moe
