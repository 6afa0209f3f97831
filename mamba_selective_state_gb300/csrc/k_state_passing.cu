// k_state_passing.cu -- cross-chunk state passing as a single-pass associative
// scan (forward and reverse), HBM-bound.
//
// Page "B200 Helion Mamba-2" (aitrends.kr/articles/109906), section "Helion
// based B200 kernel redesign": the sequential chunk loops of the forward and
// backward state passing are replaced by an associative scan.  Page
// "llm-mamba-200" (gigipick.blogspot.com), section 2: the pairs (a, b) of the
// recurrence h <- a h + b combine associatively,
//     (a, b) o (a', b') = (a a', a' b + b'),
// so the carry-in state of every chunk is an exclusive prefix of the pairs
// (a_c, S_c) applied to the initial state.
//
// Forward:   H_in[0] = init (or 0),   H_in[c+1] = a_c H_in[c] + S_c,   final = H_in[nc]
// Backward:  G[nc] = dfinal (or 0),   G[c] = dHloc[c] + a_c G[c+1],
//            dS[c] = G[c+1],          dinit = G[0]
// (dS goes to its own buffer; dHloc is read once).
// The backward is the same scan run over the chunks in reverse order.
//
// Decomposition.  A tile is (row b, head h, a block of 512 consecutive state
// elements, a segment of consecutive chunks: 16 forward, 8 in reverse).  One
// thread issues bulk asynchronous copies of the segment's chunk blocks (2 KB
// each; in reverse also the fp32 carry-in states) into shared memory, so the
// whole segment is in flight at once without holding registers; each thread
// then owns 4 consecutive elements (one float4, conflict-free in shared
// memory, coalesced in global memory) and scans the segment sequentially in
// place -- work-efficient.  Segments are joined by a look-back over
// published per-segment aggregates (the product of the decays, the locally
// scanned state), decoupled from the predecessors' own joins: every
// kSpSpan-th segment is a checkpoint that publishes its inclusive prefix;
// any other segment publishes its aggregate as soon as its local scan is
// done and then folds, in chunk order, the aggregates back to the nearest
// checkpoint before it.  The fold order is fixed, so the result does not
// depend on which predecessor happened to finish first: every run gives the
// same bits.  Only checkpoints wait on a predecessor's join, so the serial
// chain is nseg / kSpSpan long.  Tiles take their index from an atomic
// ticket, so every tile a tile waits on is already resident: the waits always
// end.  Each wait is also bounded in time; on expiry the tile records a
// timeout in the status word and continues instead of hanging.
#include "ssd_internal.cuh"
#include "tc_common.cuh"

namespace ssd {

namespace {

constexpr unsigned long long kWaitLimitNs = 2000000000ull;      // 2 s
constexpr unsigned long long kTestWaitLimitNs = 100000000ull;   // 0.1 s

__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ int ld_acquire(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release(int* p, int v) {
  asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ float4 fma4(float a, float4 x, float4 y) {
  return make_float4(fmaf(a, x.x, y.x), fmaf(a, x.y, y.y), fmaf(a, x.z, y.z), fmaf(a, x.w, y.w));
}

enum : int { kFlagNone = 0, kFlagAggregate = 1, kFlagPrefix = 2 };
constexpr int kSpSpan = 8;  // segments from one checkpoint to the next
static_assert(kSpSpan <= 32 && kSpThreads >= 96, "look-back waits use warp 1, decays warp 2");

// Public state tensors are (b, H, P, N); the chunk-state layout is (N, P):
// the 4 consecutive elements e..e+3 (same n, headdim p..p+3) of a thread map
// to public offsets (p+i)*N + n.
__device__ __forceinline__ float4 load_public(const float* base, int e, int P, int N) {
  const int n = e / P, pp = e - n * P;
  return make_float4(base[(pp + 0) * N + n], base[(pp + 1) * N + n], base[(pp + 2) * N + n],
                     base[(pp + 3) * N + n]);
}
__device__ __forceinline__ void store_public(float* base, int e, int P, int N, float4 v) {
  const int n = e / P, pp = e - n * P;
  base[(pp + 0) * N + n] = v.x;
  base[(pp + 1) * N + n] = v.y;
  base[(pp + 2) * N + n] = v.z;
  base[(pp + 3) * N + n] = v.w;
}
__device__ __forceinline__ void store4(float* dst, float4 v) { *reinterpret_cast<float4*>(dst) = v; }
__device__ __forceinline__ void store4(__nv_bfloat16* dst, float4 v) {
  __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y), b = __floats2bfloat162_rn(v.z, v.w);
  uint2 u;
  u.x = *reinterpret_cast<uint32_t*>(&a);
  u.y = *reinterpret_cast<uint32_t*>(&b);
  *reinterpret_cast<uint2*>(dst) = u;
}

// Outputs (carry-in states forward, dS backward) are written in the problem
// dtype TOut; the scan itself runs in fp32.
// kKeepF32 (forward only): also store the fp32 carry-in states over the chunk
// states just read.  The backward also forms dL/da_c = <dS_c, H_in[c]> in
// fp32 from those fp32 carry-in states: one partial per (chunk, element
// block), folded over the block's warps in a fixed order.
template <bool kBwd>
__host__ __device__ constexpr int sp_seg() { return kBwd ? kSpSegB : kSpSegF; }
template <bool kBwd>
__host__ __device__ constexpr size_t sp_smem_bytes() { return (size_t)sp_seg<kBwd>() * kSpElems * 4 * (kBwd ? 2 : 1); }

// kShfl (forward only; SSD_SCAN_WARP_SHUFFLE): the segment's local scans
// run across lanes instead of inside a thread -- lane k of a group of kSeg
// lanes holds chunk k of one float4 of elements, and log2(kSeg) Hillis-Steele
// steps of warp shuffles compose the pairs (a, b) o (a', b') = (a a', a' b + b')
// -- with the per-thread aggregates and prefixes staged through shared memory
// for the join.  Kept for comparison with the in-thread sequential scan.
template <bool kBwd, bool kKeepF32, typename TOut, bool kShfl = false>
__global__ void __launch_bounds__(kSpThreads, 3) state_passing_kernel(Plan p, Bufs f) {
  static_assert(!(kShfl && kBwd), "the warp-shuffle variant is forward only");
  constexpr int kSeg = sp_seg<kBwd>();
  extern __shared__ __align__(128) float s_buf[];  // [kSeg][kSpElems] inputs; reverse: then [kSeg][kSpElems] H_in
  __shared__ __align__(8) uint64_t s_bar;
  __shared__ int s_ticket, s_timeout;
  __shared__ float s_A[kSpSpan];  // decay products of the folded segments
  __shared__ float s_a[kSeg];     // decays of this segment's chunks, in scan order
  __shared__ float s_da[kSeg][kSpThreads / 32];
  int* flags = kBwd ? f.flags_bwd : f.flags_fwd;
  const int nseg = kBwd ? p.sp_nseg_b : p.sp_nseg;
  if (threadIdx.x == 0) {
    s_ticket = atomicAdd(kBwd ? &f.hdr->ticket_bwd : &f.hdr->ticket_fwd, 1);
    s_timeout = 0;
    tc::mbar_init(&s_bar, 1);
    tc::mbar_fence_init();
  }
  __syncthreads();
  const int ticket = s_ticket;
  const int seg = ticket / p.sp_chains;
  const int chain = ticket - seg * p.sp_chains;
  const int eblk = chain % p.sp_neblk;
  const long long bh = chain / p.sp_neblk;  // bi * H + h
  const int e0 = eblk * kSpElems;
  const int ne = min(kSpElems, p.PN - e0);  // elements of this block (a multiple of 256)
  const int e = e0 + threadIdx.x * 4;
  const bool active = e < p.PN;
  const int k0 = seg * kSeg;
  const int nk = min(kSeg, p.nc - k0);
  const float* achunk = f.achunk + bh * p.nc;
  const float* in = kBwd ? f.dHl : f.S;  // forward: chunk states; backward: dHloc
  TOut* out = static_cast<TOut*>(kBwd ? f.dS : f.Hin);
  const unsigned long long limit =
      (p.flags & SSD_TEST_DROP_SCAN_PUBLISH) ? kTestWaitLimitNs : kWaitLimitNs;
  auto chunk_of = [&](int k) { return kBwd ? p.nc - 1 - k : k; };  // k-th chunk in scan order
  auto slot_of = [&](int sg) { return ((size_t)chain * nseg + sg) * kSpElems + threadIdx.x * 4; };
  auto state_off = [&](int k) { return ((size_t)bh * p.nc + chunk_of(k0 + k)) * p.PN + e0; };

  // 1) the segment's blocks into shared memory; then the segment's aggregate
  //    (a local scan from a zero state; it is redone in step 3, where the
  //    value entering each chunk is needed, instead of being stored)
  if (threadIdx.x == 0) {
    const uint32_t bytes = (uint32_t)ne * 4u;
    tc::mbar_expect_tx(&s_bar, bytes * nk * (kBwd ? 2u : 1u));
    for (int k = 0; k < nk; ++k) {
      tc::bulk_load(s_buf + k * kSpElems, in + state_off(k), bytes, &s_bar);
      if (kBwd) tc::bulk_load(s_buf + (kSeg + k) * kSpElems, f.S + state_off(k), bytes, &s_bar);
    }
  }
  if (threadIdx.x < nk) s_a[threadIdx.x] = __ldg(achunk + chunk_of(k0 + threadIdx.x));
  __syncthreads();
  if (!tc::mbar_wait(&s_bar, 0)) atomicOr(&f.hdr->status, kDevTimeout);
  float4* vb = reinterpret_cast<float4*>(s_buf) + threadIdx.x;  // block k at vb[k * kSpThreads]
  float4 run = make_float4(0.f, 0.f, 0.f, 0.f);
  float aprod = 1.0f;
  constexpr int kBatch = kSeg < 8 ? kSeg : 8;  // loads issued together: only the FMA chain is serial
  // warp-shuffle variant: lane layout and the decay windows of each step
  constexpr int kGp = 32 / kSeg;  // float4 groups per warp pass
  const int lane = threadIdx.x & 31, wbase = threadIdx.x & ~31;
  const int kl = lane % kSeg, hl = lane / kSeg;
  __shared__ float4 s_x4[kShfl ? kSpThreads : 1];  // per-thread aggregate, then prefix
  if constexpr (kShfl) {
    const float4* v4 = reinterpret_cast<const float4*>(s_buf);
    const float a0 = kl < nk ? s_a[kl] : 1.0f;
    for (int pass = 0; pass < 32 / kGp; ++pass) {
      const int g = wbase + pass * kGp + hl;  // float4 group of this lane
      float4 b = (kl < nk && e0 + g * 4 < p.PN) ? v4[kl * kSpThreads + g] : make_float4(0.f, 0.f, 0.f, 0.f);
      float a = a0;
#pragma unroll
      for (int d = 1; d < kSeg; d <<= 1) {
        const float ao = __shfl_up_sync(0xffffffffu, a, d, kSeg);
        const float4 bo = make_float4(__shfl_up_sync(0xffffffffu, b.x, d, kSeg), __shfl_up_sync(0xffffffffu, b.y, d, kSeg),
                                      __shfl_up_sync(0xffffffffu, b.z, d, kSeg), __shfl_up_sync(0xffffffffu, b.w, d, kSeg));
        if (kl >= d) {
          b = fma4(a, bo, b);
          a *= ao;
        }
      }
      if (kl == nk - 1) {
        s_x4[g] = b;
        if (g == wbase) s_A[0] = a;  // the segment's decay product (every lane of chunk nk-1 agrees)
      }
    }
    __syncthreads();
    run = s_x4[threadIdx.x];
    aprod = s_A[0];
    __syncthreads();  // s_A is reused by the join
  }
#pragma unroll
  for (int kb = 0; kb < (kShfl ? 0 : kSeg); kb += kBatch) {
    float4 x[kBatch];
#pragma unroll
    for (int k = 0; k < kBatch; ++k)
      x[k] = (kb + k < nk && active) ? vb[(kb + k) * kSpThreads] : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int k = 0; k < kBatch; ++k) {
      if (kb + k < nk) {
        run = fma4(s_a[kb + k], run, x[k]);
        aprod *= s_a[kb + k];
      }
    }
  }

  // 2) join with the predecessors
  const bool is_check = seg % kSpSpan == 0;
  const bool drop = (p.flags & SSD_TEST_DROP_SCAN_PUBLISH) && seg == 0 && chain == 0;
  float4 prefix = make_float4(0.f, 0.f, 0.f, 0.f);
  if (!is_check && seg + 1 < nseg) {  // publish the aggregate at once
    if (active) __stcg(reinterpret_cast<float4*>(f.agg + slot_of(seg)), run);
    __syncthreads();  // every thread's part is written; one release (cumulative) publishes them all
    if (threadIdx.x == 0) st_release(flags + (size_t)chain * nseg + seg, kFlagAggregate);
  }
  if (seg == 0) {
    const float* start = kBwd ? f.dfinal : f.init;
    if (start != nullptr && active) prefix = load_public(start + bh * p.PN, e, p.P, p.N);
  } else {
    // the nearest checkpoint before this segment, and the segments between
    const int anchor = is_check ? seg - kSpSpan : (seg / kSpSpan) * kSpSpan;
    const int nfold = seg - anchor - 1;
    // lane t of warp 1 waits for segment anchor + t (warp 0 may still be
    // releasing this tile's aggregate; warp 2 reads the decays meanwhile)
    const int tw = (int)threadIdx.x - 32;
    if (tw >= 0 && tw <= nfold) {
      const int* fp = flags + (size_t)chain * nseg + anchor + tw;
      if (ld_acquire(fp) == kFlagNone) {
        const unsigned long long t_start = global_ns();
        const long long c_start = clock64();
        unsigned polls = 0;
        while (ld_acquire(fp) == kFlagNone) {
          if (global_ns() - t_start > limit || clock64() - c_start > 2 * (long long)limit ||
              ++polls > (1u << 24)) {
            atomicOr(&f.hdr->status, kDevTimeout);
            s_timeout = 1;
            break;
          }
          __nanosleep(128);
        }
      }
    }
    const int ta = (int)threadIdx.x - 64;
    if (ta >= 0 && ta < nfold) {  // decay product of segment anchor + 1 + t, in chunk order
      const int sg = anchor + 1 + ta;
      float a = 1.0f;
      for (int k = 0; k < kSeg; ++k) a *= __ldg(achunk + chunk_of(sg * kSeg + k));
      s_A[ta] = a;
    }
    __syncthreads();
    if (active && !s_timeout) {  // every load first, then the fold in chunk order
      prefix = __ldcg(reinterpret_cast<const float4*>(f.incl + slot_of(anchor)));
      float4 bk[kSpSpan - 1];
#pragma unroll
      for (int t = 0; t < kSpSpan - 1; ++t)
        if (t < nfold) bk[t] = __ldcg(reinterpret_cast<const float4*>(f.agg + slot_of(anchor + 1 + t)));
#pragma unroll
      for (int t = 0; t < kSpSpan - 1; ++t)
        if (t < nfold) prefix = fma4(s_A[t], prefix, bk[t]);
    }
  }
  const float4 incl = fma4(aprod, prefix, run);
  if (is_check && seg + 1 < nseg && !drop) {  // checkpoints publish their inclusive prefix
    if (active) __stcg(reinterpret_cast<float4*>(f.incl + slot_of(seg)), incl);
    __syncthreads();  // every thread's part is written; one release (cumulative) publishes them all
    if (threadIdx.x == 0) st_release(flags + (size_t)chain * nseg + seg, kFlagPrefix);
  }

  // 3) carry-in values of the segment's chunks, and the end of the chain
  float dp = 1.0f;  // product of the decays before chunk k (same order as aprod)
  float4 loc = make_float4(0.f, 0.f, 0.f, 0.f);  // the local scan again: value entering chunk k
  if constexpr (kShfl) {
    // the value entering chunk k: the exclusive scan (lane k-1's inclusive
    // pair) applied to the segment's entering state
    s_x4[threadIdx.x] = prefix;
    __syncthreads();
    const float4* v4 = reinterpret_cast<const float4*>(s_buf);
    const float a0 = kl < nk ? s_a[kl] : 1.0f;
    for (int pass = 0; pass < 32 / kGp; ++pass) {
      const int g = wbase + pass * kGp + hl;
      const bool gact = e0 + g * 4 < p.PN;
      float4 b = (kl < nk && gact) ? v4[kl * kSpThreads + g] : make_float4(0.f, 0.f, 0.f, 0.f);
      float a = a0;
#pragma unroll
      for (int d = 1; d < kSeg; d <<= 1) {
        const float ao = __shfl_up_sync(0xffffffffu, a, d, kSeg);
        const float4 bo = make_float4(__shfl_up_sync(0xffffffffu, b.x, d, kSeg), __shfl_up_sync(0xffffffffu, b.y, d, kSeg),
                                      __shfl_up_sync(0xffffffffu, b.z, d, kSeg), __shfl_up_sync(0xffffffffu, b.w, d, kSeg));
        if (kl >= d) {
          b = fma4(a, bo, b);
          a *= ao;
        }
      }
      float ae = __shfl_up_sync(0xffffffffu, a, 1, kSeg);
      float4 be = make_float4(__shfl_up_sync(0xffffffffu, b.x, 1, kSeg), __shfl_up_sync(0xffffffffu, b.y, 1, kSeg),
                              __shfl_up_sync(0xffffffffu, b.z, 1, kSeg), __shfl_up_sync(0xffffffffu, b.w, 1, kSeg));
      if (kl == 0) {
        ae = 1.0f;
        be = make_float4(0.f, 0.f, 0.f, 0.f);
      }
      if (kl < nk && gact) {
        const size_t off = state_off(kl) + g * 4;
        const float4 val = fma4(ae, s_x4[g], be);
        store4(out + off, val);
        if (kKeepF32) __stcs(reinterpret_cast<float4*>(f.S + off), val);
      }
    }
  }
#pragma unroll
  for (int kb = 0; kb < (kShfl ? 0 : kSeg); kb += kBatch) {
   float4 x[kBatch];
#pragma unroll
   for (int k2 = 0; k2 < kBatch; ++k2)
     x[k2] = (kb + k2 < nk && active) ? vb[(kb + k2) * kSpThreads] : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
   for (int k2 = 0; k2 < kBatch; ++k2) {
    const int k = kb + k2;
    if (k >= nk) break;
    const size_t off = state_off(k) + threadIdx.x * 4;
    const float4 val = fma4(dp, prefix, loc);
    loc = fma4(s_a[k], loc, x[k2]);
    dp *= s_a[k];
    if (active) {
      store4(out + off, val);
      if (kKeepF32) __stcs(reinterpret_cast<float4*>(f.S + off), val);
    }
    if (kBwd) {
      float d = 0.0f;
      if (active) {
        const float4 h4 = vb[(kSeg + k) * kSpThreads];
        d = val.x * h4.x + val.y * h4.y + val.z * h4.z + val.w * h4.w;
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) d += __shfl_xor_sync(0xffffffffu, d, o);
      if ((threadIdx.x & 31) == 0) s_da[k][threadIdx.x >> 5] = d;
    }
   }
  }
  if (kBwd) {
    __syncthreads();
    if (threadIdx.x < nk) {
      const int k = threadIdx.x;
      float d = 0.0f;
      for (int w = 0; w < kSpThreads / 32; ++w) d += s_da[k][w];
      f.dapart[((size_t)bh * p.nc + chunk_of(k0 + k)) * p.da_stride + eblk] = d;
    }
  }
  if (active) {
    if (seg == nseg - 1) {
      float* fin = kBwd ? f.dinit : f.final_states;
      if (fin != nullptr) store_public(fin + bh * p.PN, e, p.P, p.N, incl);
    }
  }
}

template <bool kBwd, bool kKeepF32, typename TOut>
cudaError_t launch_sp(const Plan& p, const Bufs& f, cudaStream_t s) {
  const unsigned tiles = (unsigned)p.sp_chains * (kBwd ? p.sp_nseg_b : p.sp_nseg);
  auto kern = state_passing_kernel<kBwd, kKeepF32, TOut>;
  if constexpr (!kBwd)
    if (p.flags & SSD_SCAN_WARP_SHUFFLE) kern = state_passing_kernel<kBwd, kKeepF32, TOut, true>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)sp_smem_bytes<kBwd>());
  if (e != cudaSuccess) return e;
  kern<<<tiles, kSpThreads, sp_smem_bytes<kBwd>(), s>>>(p, f);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_state_passing(const Plan& p, const Bufs& f, bool backward, bool keep_f32, cudaStream_t s) {
  set_kernel_name(backward ? "state_passing_bwd" : (keep_f32 ? "state_passing_fwd_keep" : "state_passing_fwd"));
  const bool bf = p.dtype == SSD_BF16;
  if (backward) return bf ? launch_sp<true, false, __nv_bfloat16>(p, f, s) : launch_sp<true, false, float>(p, f, s);
  if (keep_f32) return bf ? launch_sp<false, true, __nv_bfloat16>(p, f, s) : launch_sp<false, true, float>(p, f, s);
  return bf ? launch_sp<false, false, __nv_bfloat16>(p, f, s) : launch_sp<false, false, float>(p, f, s);
}

}  // namespace ssd
