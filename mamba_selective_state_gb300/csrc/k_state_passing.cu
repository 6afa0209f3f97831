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
// Decomposition.  A tile is (row b, head h, a block of 1024 consecutive state
// elements, a segment of kSpSeg consecutive chunks).  Each thread owns 4
// consecutive elements (one float4, coalesced across the CTA) and scans its
// segment sequentially -- work-efficient; the loads do not depend on the
// carry and are all issued up front.  Segments are joined by a look-back
// over published per-segment aggregates (the product of the decays, the
// locally scanned state), decoupled from the predecessors' own joins: every
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
// states just read (each element is read before it is written, by the same
// thread).  The backward also forms dL/da_c = <dS_c, H_in[c]> in fp32 from
// those fp32 carry-in states: one partial per (chunk, element block), folded
// over the block's warps in a fixed order.
template <bool kBwd, bool kKeepF32, typename TOut>
__global__ void __launch_bounds__(kSpThreads, kBwd ? 2 : 4) state_passing_kernel(Plan p, Bufs f) {
  __shared__ int s_ticket, s_timeout;
  __shared__ float s_A[kSpSpan];  // decay products of the folded segments
  __shared__ float s_da[kSpSeg][kSpThreads / 32];
  int* flags = kBwd ? f.flags_bwd : f.flags_fwd;
  if (threadIdx.x == 0) {
    s_ticket = atomicAdd(kBwd ? &f.hdr->ticket_bwd : &f.hdr->ticket_fwd, 1);
    s_timeout = 0;
  }
  __syncthreads();
  const int ticket = s_ticket;
  const int seg = ticket / p.sp_chains;
  const int chain = ticket - seg * p.sp_chains;
  const int eblk = chain % p.sp_neblk;
  const long long bh = chain / p.sp_neblk;  // bi * H + h
  const int e = eblk * kSpElems + threadIdx.x * 4;
  const bool active = e < p.PN;
  const int k0 = seg * kSpSeg;
  const int nk = min(kSpSeg, p.nc - k0);
  const float* achunk = f.achunk + bh * p.nc;
  const float* in = kBwd ? f.dHl : f.S;  // forward: chunk states; backward: dHloc
  TOut* out = static_cast<TOut*>(kBwd ? f.dS : f.Hin);
  const unsigned long long limit =
      (p.flags & SSD_TEST_DROP_SCAN_PUBLISH) ? kTestWaitLimitNs : kWaitLimitNs;
  auto chunk_of = [&](int k) { return kBwd ? p.nc - 1 - k : k; };  // k-th chunk in scan order
  auto slot_of = [&](int sg) { return ((size_t)chain * p.sp_nseg + sg) * kSpElems + threadIdx.x * 4; };
  auto state_off = [&](int k) { return ((size_t)bh * p.nc + chunk_of(k0 + k)) * p.PN + e; };

  // 1) local scan of the segment from a zero state; v[k] becomes the value
  //    entering chunk k, dprod[k] the product of the decays before chunk k.
  float4 v[kSpSeg];
  float dprod[kSpSeg];
#pragma unroll
  for (int k = 0; k < kSpSeg; ++k) {
    v[k] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (k < nk && active) v[k] = __ldcs(reinterpret_cast<const float4*>(in + state_off(k)));
  }
  // backward: the fp32 carry-in states of the segment's chunks, for dL/da_c
  // at the end (loaded now, so that their latency hides under the join)
  float4 hv[kBwd ? kSpSeg : 1];
#pragma unroll
  for (int k = 0; k < (kBwd ? kSpSeg : 0); ++k) {
    hv[k] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (k < nk && active) hv[k] = __ldcs(reinterpret_cast<const float4*>(f.S + state_off(k)));
  }
  float4 run = make_float4(0.f, 0.f, 0.f, 0.f);
  float aprod = 1.0f;
#pragma unroll
  for (int k = 0; k < kSpSeg; ++k) {
    if (k < nk) {
      const float a = __ldg(achunk + chunk_of(k0 + k));
      const float4 x = v[k];
      v[k] = run;
      dprod[k] = aprod;
      run = fma4(a, run, x);
      aprod *= a;
    }
  }

  // 2) join with the predecessors
  const bool is_check = seg % kSpSpan == 0;
  const bool drop = (p.flags & SSD_TEST_DROP_SCAN_PUBLISH) && seg == 0 && chain == 0;
  float4 prefix = make_float4(0.f, 0.f, 0.f, 0.f);
  if (!is_check && seg + 1 < p.sp_nseg) {  // publish the aggregate at once
    if (active) __stcg(reinterpret_cast<float4*>(f.agg + slot_of(seg)), run);
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) st_release(flags + (size_t)chain * p.sp_nseg + seg, kFlagAggregate);
  }
  if (seg == 0) {
    const float* start = kBwd ? f.dfinal : f.init;
    if (start != nullptr && active) prefix = load_public(start + bh * p.PN, e, p.P, p.N);
  } else {
    // the nearest checkpoint before this segment, and the segments between
    const int anchor = is_check ? seg - kSpSpan : (seg / kSpSpan) * kSpSpan;
    const int nfold = seg - anchor - 1;
    if (threadIdx.x <= nfold) {  // thread t waits for segment anchor + t
      const int* fp = flags + (size_t)chain * p.sp_nseg + anchor + threadIdx.x;
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
      __threadfence();
    }
    if (threadIdx.x < nfold) {  // decay product of segment anchor + 1 + t, in chunk order
      const int sg = anchor + 1 + threadIdx.x;
      float a = 1.0f;
      for (int k = 0; k < kSpSeg; ++k) a *= __ldg(achunk + chunk_of(sg * kSpSeg + k));
      s_A[threadIdx.x] = a;
    }
    __syncthreads();
    if (active && !s_timeout) {
      prefix = __ldcg(reinterpret_cast<const float4*>(f.incl + slot_of(anchor)));
#pragma unroll 1
      for (int t = 0; t < nfold; ++t) {
        const float4 bk = __ldcg(reinterpret_cast<const float4*>(f.agg + slot_of(anchor + 1 + t)));
        prefix = fma4(s_A[t], prefix, bk);
      }
    }
  }
  const float4 incl = fma4(aprod, prefix, run);
  if (is_check && seg + 1 < p.sp_nseg && !drop) {  // checkpoints publish their inclusive prefix
    if (active) __stcg(reinterpret_cast<float4*>(f.incl + slot_of(seg)), incl);
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) st_release(flags + (size_t)chain * p.sp_nseg + seg, kFlagPrefix);
  }

  // 3) carry-in values of the segment's chunks, and the end of the chain
#pragma unroll
  for (int k = 0; k < kSpSeg; ++k) {
    if (k < nk) {
      const size_t off = state_off(k);
      const float4 val = fma4(dprod[k], prefix, v[k]);
      if (active) {
        store4(out + off, val);
        if (kKeepF32) *reinterpret_cast<float4*>(f.S + off) = val;
      }
      if (kBwd) {
        const float4 h4 = hv[k];
        float d = val.x * h4.x + val.y * h4.y + val.z * h4.z + val.w * h4.w;
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
      f.dapart[((size_t)bh * p.nc + chunk_of(k0 + k)) * p.sp_neblk + eblk] = d;
    }
  }
  if (active) {
    if (seg == p.sp_nseg - 1) {
      float* fin = kBwd ? f.dinit : f.final_states;
      if (fin != nullptr) store_public(fin + bh * p.PN, e, p.P, p.N, incl);
    }
  }
}

}  // namespace

cudaError_t launch_state_passing(const Plan& p, const Bufs& f, bool backward, bool keep_f32, cudaStream_t s) {
  const unsigned tiles = (unsigned)p.sp_chains * p.sp_nseg;
  set_kernel_name(backward ? "state_passing_bwd" : (keep_f32 ? "state_passing_fwd_keep" : "state_passing_fwd"));
  const bool bf = p.dtype == SSD_BF16;
  if (backward) {
    if (bf) state_passing_kernel<true, false, __nv_bfloat16><<<tiles, kSpThreads, 0, s>>>(p, f);
    else state_passing_kernel<true, false, float><<<tiles, kSpThreads, 0, s>>>(p, f);
  } else if (keep_f32) {
    if (bf) state_passing_kernel<false, true, __nv_bfloat16><<<tiles, kSpThreads, 0, s>>>(p, f);
    else state_passing_kernel<false, true, float><<<tiles, kSpThreads, 0, s>>>(p, f);
  } else {
    if (bf) state_passing_kernel<false, false, __nv_bfloat16><<<tiles, kSpThreads, 0, s>>>(p, f);
    else state_passing_kernel<false, false, float><<<tiles, kSpThreads, 0, s>>>(p, f);
  }
  return cudaGetLastError();
}

}  // namespace ssd
