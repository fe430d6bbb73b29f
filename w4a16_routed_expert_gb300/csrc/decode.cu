// Decode megakernel: the whole layer forward for a small batch (T <= 16,
// fully resident table) in one cooperative launch, one CTA per SM.
//
// The multi-kernel path pays a launch boundary and a pipeline ramp between
// routing, gate/up, down and the combine; at batch 1 each of those costs as
// much as streaming the weights. Here, inside one persistent grid whose CTAs
// are all resident (cooperative launch):
//   1. router logits: one expert row per warp across the whole grid;
//   2. a grid-wide arrival count on the logits; then every CTA computes the
//      top-k, the permutation and the segment list itself, into its own
//      shared memory (identical results in every CTA, no second grid hop);
//      CTA 0 also publishes them to global memory;
//   3. gate/up + SwiGLU work items (the GEMV's items); every consumer warp
//      signals a per-segment counter after its h rows are written;
//   4. down work items, whose weights the producer streams into the ring
//      while gate/up items are still being computed; a consumer warp waits
//      for its segment's gate/up counter before reading h;
//   5. every down item signals a per-row-block counter; the warp that
//      completes a row block performs the weighted combine for those rows
//      (fixed order: ranks j = 0..k-1, then the shared expert).
// Every cross-CTA wait is a bounded spin; on time-out the CTA records an
// error, stops, lets its issued copies land and still passes the final
// ticket, whose last holder resets all counters for the next launch.
#include "gemv_dev.cuh"
#include "route_dev.cuh"

namespace moe {

namespace {

struct DecodeHdr {
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  int abort_flag;
  int issued;
  int last;
};

// Release-ordered increment (fire and forget): the caller's prior writes, and
// those of the warp lanes synchronised with it, are visible before it.
__device__ __forceinline__ void red_release_add(uint32_t* p, uint32_t v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t atom_acq_rel_add(uint32_t* p, uint32_t v) {
  uint32_t old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

__device__ __forceinline__ uint32_t ld_acquire(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Bounded spin until *p >= target. False on time-out (error recorded).
__device__ __forceinline__ bool wait_count(const uint32_t* p, uint32_t target, volatile int* abort_flag,
                                           uint32_t* err) {
  if (ld_acquire(p) >= target) return true;
  const long long t0 = clock64();
  while (true) {
    __nanosleep(64);
    if (ld_acquire(p) >= target) return true;
    if (*abort_flag) return false;
    if (clock64() - t0 > kSpinLimitCycles) {
      record_error(err, MOE_DEV_ERR_TIMEOUT);
      *abort_flag = 1;
      return false;
    }
  }
}

template <int NV, int KG, int NTG, int KD, int NTD>
__global__ void __launch_bounds__(kGemvThreads, 1) k_decode(DecodeArgs a) {
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ int s_scan[33];
  DecodeHdr* hdr = reinterpret_cast<DecodeHdr*>(smem);
  unsigned char* ring = smem + kHdrBytes;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int S = a.stages;
  const int T = a.r.T, H = a.r.H, E = a.r.E, k = a.r.k;
  const int Tk = T * k;
  uint32_t* logits_done = a.ctr;
  uint32_t* final_ticket = a.ctr + 1;
  uint32_t* done_gu = a.ctr + 2;
  uint32_t* done_dn = a.ctr + 2 + (E + 1);

  // routing results of this CTA, in shared memory
  int32_t* rs = reinterpret_cast<int32_t*>(ring + (size_t)S * a.slot_bytes);
  int32_t* s_ids = rs;                 // [Tk]
  float* s_w = reinterpret_cast<float*>(s_ids + 512);
  int32_t* s_counts = s_ids + 1024;    // [E]
  int32_t* s_off = s_counts + 1024;    // [E+1]
  int32_t* s_perm = s_off + 1025;      // [Tk]
  int32_t* s_inv = s_perm + 512;       // [Tk]
  int32_t* s_sexp = s_inv + 512;       // [E+1]
  int32_t* s_sstart = s_sexp + 1025;   // [E+1]
  int32_t* s_scount = s_sstart + 1025; // [E+1]
  int32_t* s_nseg = s_scount + 1025;   // [1]
  int32_t* s_scratch = s_nseg + 4;     // [Tk + 3E + 66]

  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&hdr->full[s], 1);
      mbar_init(&hdr->empty[s], kConsumerWarps);
    }
    hdr->abort_flag = 0;
    hdr->issued = 0;
    hdr->last = 0;
    fence_mbar_init();
  }
  __syncthreads();
  volatile int* abort_flag = &hdr->abort_flag;

  // ------------------------------------------------ 1. router logits (FP32)
  {
    const int nw = gridDim.x * (kGemvThreads / 32);
    for (int e = warp * gridDim.x + blockIdx.x; e < E; e += nw) warp_expert_logits(a.r, e);
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    atomicAdd(logits_done, 1u);
    wait_count(logits_done, gridDim.x, abort_flag, a.r.err);
  }
  __syncthreads();

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
    route_finish_cta<NV>(L, s_scratch, s_scan);
    __syncthreads();
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
  GemvArgs g = a.g, d = a.d;
  g.seg_expert = d.seg_expert = s_sexp;
  g.seg_start = d.seg_start = s_sstart;
  g.seg_count = d.seg_count = s_scount;
  g.perm = d.perm = s_perm;
  const int nrb_g = (g.N + g.rb - 1) / g.rb;
  const int nrb_d = (d.N + d.rb - 1) / d.rb;
  const int tot_g = nseg * nrb_g, tot_d = nseg * nrb_d;
  const int ipc_g = (tot_g + gridDim.x - 1) / gridDim.x, ipc_d = (tot_d + gridDim.x - 1) / gridDim.x;
  const int fg = blockIdx.x * ipc_g, fd = blockIdx.x * ipc_d;
  const int ng_it = max(0, min(tot_g, fg + ipc_g) - fg);
  const int nd_it = max(0, min(tot_d, fd + ipc_d) - fd);
  const int n_it = *abort_flag ? 0 : ng_it + nd_it;
  const uint32_t gu_target = (uint32_t)nrb_g * kConsumerWarps;
  const uint32_t dn_target = (uint32_t)nseg * kConsumerWarps;

  if (warp == kConsumerWarps) {
    if (lane == 0) {
      const uint64_t pol = l2_policy_evict_first();
      for (int it = 0; it < n_it; ++it) {
        const int st = it % S;
        const uint32_t ph = (uint32_t)(it / S) & 1u;
        if (!mbar_wait(&hdr->empty[st], ph ^ 1u, abort_flag, a.r.err)) break;
        unsigned char* slot = ring + (size_t)st * a.slot_bytes;
        if (it < ng_it)
          gemv_issue_item<true>(g, fg + it, nrb_g, slot, &hdr->full[st], pol);
        else
          gemv_issue_item<false>(d, fd + it - ng_it, nrb_d, slot, &hdr->full[st], pol);
        hdr->issued = it + 1;
      }
    }
  } else {
    XRegs<KG, NTG> xg;
    XRegs<KD, NTD> xd;
    for (int it = 0; it < n_it; ++it) {
      const int st = it % S;
      const uint32_t ph = (uint32_t)(it / S) & 1u;
      if (!mbar_wait(&hdr->full[st], ph, abort_flag, a.r.err)) break;
      const unsigned char* slot = ring + (size_t)st * a.slot_bytes;
      if (it < ng_it) {
        const int item = fg + it;
        gemv_consume_item<KG, NTG, true, false>(g, item, nrb_g, slot, xg, warp, lane);
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&hdr->empty[st]);
          red_release_add(done_gu + item / nrb_g, 1u);
        }
      } else {
        const int item = fd + it - ng_it;
        const int sgi = item / nrb_d, rbi = item % nrb_d;
        int ok = 1;
        if (lane == 0) ok = wait_count(done_gu + sgi, gu_target, abort_flag, a.r.err);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        gemv_consume_item<KD, NTD, false, true>(d, item, nrb_d, slot, xd, warp, lane);
        __syncwarp();
        uint32_t prev = 0;
        if (lane == 0) {
          mbar_arrive(&hdr->empty[st]);
          prev = atom_acq_rel_add(done_dn + rbi, 1u);
        }
        prev = __shfl_sync(0xffffffffu, prev, 0);
        if (prev + 1 == dn_target) {
          // ------------------------------- 5. combine of this row block
          // (lane 0's acq_rel increment observed every other warp's release)
          __syncwarp();
          const int r0 = rbi * d.rb;
          const int nrows = min(d.rb, H - r0);
          for (int r = lane; r < nrows; r += 32) {
            const int row = r0 + r;
            for (int t = 0; t < T; ++t) {
              float acc = 0.f;
              for (int j = 0; j < k; ++j)
                acc = fmaf(s_w[t * k + j], __ldcg(d.y_out + (size_t)(t * k + j) * H + row), acc);
              if (a.has_shared) acc += __ldcg(d.y_out + (size_t)(Tk + t) * H + row);
              __half o = __float2half_rn(acc);
              if (a.x_res) o = __float2half_rn(__half2float(a.x_res[(size_t)t * H + row]) + __half2float(o));
              a.out[(size_t)t * H + row] = o;
            }
          }
        }
      }
    }
  }

  // ---------------------------------------------------------------- teardown
  __syncthreads();
  if (tid == 0 && hdr->abort_flag) {
    const int issued = hdr->issued;
    for (int s = 0; s < S && s < issued; ++s) {
      const int n = (issued - 1 - s) / S;
      mbar_wait(&hdr->full[s], (uint32_t)n & 1u, nullptr, nullptr);
    }
  }
  if (tid == 0) {
    __threadfence();
    hdr->last = (atomicAdd(final_ticket, 1u) == gridDim.x - 1) ? 1 : 0;
  }
  __syncthreads();
  if (hdr->last) {
    // every CTA has finished: reset the counters for the next launch
    __threadfence();
    for (int i = tid; i <= E; i += blockDim.x) done_gu[i] = 0u;
    for (int i = tid; i < nrb_d; i += blockDim.x) done_dn[i] = 0u;
    if (tid == 0) {
      *logits_done = 0u;
      *final_ticket = 0u;
    }
  }
}

template <int NV, int KG, int NTG, int KD, int NTD>
cudaError_t launch_decode_t(const DecodeArgs& a, int grid, cudaStream_t s) {
  const size_t smem = decode_smem_bytes(a.stages, a.slot_bytes);
  cudaError_t e = ensure_smem(k_decode<NV, KG, NTG, KD, NTD>, smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kGemvThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k_decode<NV, KG, NTG, KD, NTD>, a);
}

template <int KG, int NTG, int KD, int NTD>
cudaError_t launch_decode_nv(const DecodeArgs& a, int grid, cudaStream_t s) {
  if (a.r.E <= 64) return launch_decode_t<2, KG, NTG, KD, NTD>(a, grid, s);
  if (a.r.E <= 128) return launch_decode_t<4, KG, NTG, KD, NTD>(a, grid, s);
  if (a.r.E <= 256) return launch_decode_t<8, KG, NTG, KD, NTD>(a, grid, s);
  if (a.r.E <= 512) return launch_decode_t<16, KG, NTG, KD, NTD>(a, grid, s);
  return launch_decode_t<32, KG, NTG, KD, NTD>(a, grid, s);
}

}  // namespace

size_t decode_smem_bytes(int stages, uint32_t slot_bytes) {
  // header, ring, routing arrays (8 x 1025 + 4 ints), finish scratch (512 + 3 x 1024 + 66 ints)
  return kHdrBytes + (size_t)stages * slot_bytes + (8 * 1025 + 4 + 512 + 3 * 1024 + 66) * sizeof(int32_t);
}

bool decode_supported(int kg, int ntg, int kd, int ntd) {
  return (kg == 2 && kd == 1 && ntg == 1 && (ntd == 1 || ntd == 2)) ||
         (kg == 1 && kd == 1 && ((ntg == 1 && ntd == 1) || (ntg == 2 && ntd == 2)));
}

cudaError_t launch_decode(const DecodeArgs& a, int kg, int ntg, int kd, int ntd, int grid, cudaStream_t s) {
  if (kg == 2 && kd == 1 && ntg == 1 && ntd == 1) return launch_decode_nv<2, 1, 1, 1>(a, grid, s);
  if (kg == 2 && kd == 1 && ntg == 1 && ntd == 2) return launch_decode_nv<2, 1, 1, 2>(a, grid, s);
  if (kg == 1 && kd == 1 && ntg == 1 && ntd == 1) return launch_decode_nv<1, 1, 1, 1>(a, grid, s);
  if (kg == 1 && kd == 1 && ntg == 2 && ntd == 2) return launch_decode_nv<1, 2, 1, 2>(a, grid, s);
  return cudaErrorInvalidConfiguration;
}

}  // namespace moe
