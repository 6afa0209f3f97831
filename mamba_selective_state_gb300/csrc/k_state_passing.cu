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
// segment sequentially -- work-efficient, the loads do not depend on the
// carry and are all issued up front.  Segments are joined by decoupled
// lookback: a tile publishes its aggregate pair (the product of the decays, the
// locally scanned state) as soon as it has it, then walks back over its
// predecessors, folding aggregates until it meets a published inclusive
// prefix.  Tiles take their index from an atomic ticket, so every tile a
// tile waits on is already resident: the waits always end.  Each wait is also
// bounded in time; on expiry the tile records a timeout in the status word
// and continues with a zero prefix instead of hanging.
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
__global__ void __launch_bounds__(kSpThreads) state_passing_kernel(Plan p, Bufs f) {
  __shared__ int s_ticket, s_flag;
  __shared__ float s_da[kSpSeg][kSpThreads / 32];
  int* flags = kBwd ? f.flags_bwd : f.flags_fwd;
  if (threadIdx.x == 0) s_ticket = atomicAdd(kBwd ? &f.hdr->ticket_bwd : &f.hdr->ticket_fwd, 1);
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
  const size_t lb_slot = ((size_t)chain * p.sp_nseg + seg) * kSpElems + threadIdx.x * 4;
  const unsigned long long limit =
      (p.flags & SSD_TEST_DROP_SCAN_PUBLISH) ? kTestWaitLimitNs : kWaitLimitNs;

  // 1) local scan of the segment from a zero state; v[k] becomes the value
  //    entering chunk k, dprod[k] the product of the decays before chunk k.
  float4 v[kSpSeg];
  float dprod[kSpSeg];
#pragma unroll
  for (int k = 0; k < kSpSeg; ++k) {
    v[k] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (k < nk && active) {
      const int c = kBwd ? p.nc - 1 - (k0 + k) : k0 + k;
      v[k] = __ldcs(reinterpret_cast<const float4*>(in + ((size_t)bh * p.nc + c) * p.PN + e));
    }
  }
  float4 run = make_float4(0.f, 0.f, 0.f, 0.f);
  float aprod = 1.0f;
#pragma unroll
  for (int k = 0; k < kSpSeg; ++k) {
    if (k < nk) {
      const int c = kBwd ? p.nc - 1 - (k0 + k) : k0 + k;
      const float a = __ldg(achunk + c);
      const float4 x = v[k];
      v[k] = run;
      dprod[k] = aprod;
      run = fma4(a, run, x);
      aprod *= a;
    }
  }

  // 2) join with the predecessors
  float4 prefix = make_float4(0.f, 0.f, 0.f, 0.f);
  if (seg == 0) {
    const float* start = kBwd ? f.dfinal : f.init;
    if (start != nullptr && active) prefix = load_public(start + bh * p.PN, e, p.P, p.N);
  } else {
    if (active) __stcg(reinterpret_cast<float4*>(f.agg + lb_slot), run);
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) st_release(flags + (size_t)chain * p.sp_nseg + seg, kFlagAggregate);
    float acc_a = 1.0f;
    float4 acc_v = make_float4(0.f, 0.f, 0.f, 0.f);
    int sp = seg - 1;
    bool joined = false;
    while (sp >= 0) {
      if (threadIdx.x == 0) {
        const int* fp = flags + (size_t)chain * p.sp_nseg + sp;
        int fl = ld_acquire(fp);
        if (fl == kFlagNone) {
          const unsigned long long t_start = global_ns();
          const long long c_start = clock64();
          unsigned polls = 0;
          while ((fl = ld_acquire(fp)) == kFlagNone) {
            if (global_ns() - t_start > limit || clock64() - c_start > 2 * (long long)limit ||
                ++polls > (1u << 24)) {
              atomicOr(&f.hdr->status, kDevTimeout);
              fl = -1;
              break;
            }
            __nanosleep(128);
          }
        }
        __threadfence();
        s_flag = fl;
      }
      __syncthreads();
      const int fl = s_flag;
      __syncthreads();
      if (fl < 0) break;  // timed out: continue from what has been folded so far
      const size_t slot = ((size_t)chain * p.sp_nseg + sp) * kSpElems + threadIdx.x * 4;
      if (fl == kFlagPrefix) {
        float4 pv = make_float4(0.f, 0.f, 0.f, 0.f);
        if (active) pv = __ldcg(reinterpret_cast<const float4*>(f.incl + slot));
        prefix = fma4(acc_a, pv, acc_v);
        joined = true;
        break;
      }
      // aggregate of segment sp: fold it under the spans already folded
      float4 av = make_float4(0.f, 0.f, 0.f, 0.f);
      if (active) av = __ldcg(reinterpret_cast<const float4*>(f.agg + slot));
      float a_sp = 1.0f;
      const int ks = sp * kSpSeg, kn = min(kSpSeg, p.nc - ks);
      for (int k = 0; k < kn; ++k) a_sp *= __ldg(achunk + (kBwd ? p.nc - 1 - (ks + k) : ks + k));
      acc_v = fma4(acc_a, av, acc_v);
      acc_a *= a_sp;
      --sp;
    }
    if (!joined) {
      if (sp < 0) {  // walked back to the chain start
        const float* start = kBwd ? f.dfinal : f.init;
        float4 sv = make_float4(0.f, 0.f, 0.f, 0.f);
        if (start != nullptr && active) sv = load_public(start + bh * p.PN, e, p.P, p.N);
        prefix = fma4(acc_a, sv, acc_v);
      } else {
        prefix = acc_v;  // timed out
      }
    }
  }
  const float4 incl = fma4(aprod, prefix, run);
  const bool drop = (p.flags & SSD_TEST_DROP_SCAN_PUBLISH) && seg == 0 && chain == 0;
  if (seg + 1 < p.sp_nseg && !drop) {
    if (active) __stcg(reinterpret_cast<float4*>(f.incl + lb_slot), incl);
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) st_release(flags + (size_t)chain * p.sp_nseg + seg, kFlagPrefix);
  }

  // 3) carry-in values of the segment's chunks, and the end of the chain
#pragma unroll
  for (int k = 0; k < kSpSeg; ++k) {
    if (k < nk) {
      const int c = kBwd ? p.nc - 1 - (k0 + k) : k0 + k;
      const size_t off = ((size_t)bh * p.nc + c) * p.PN + e;
      const float4 val = fma4(dprod[k], prefix, v[k]);
      if (active) {
        store4(out + off, val);
        if (kKeepF32) *reinterpret_cast<float4*>(f.S + off) = val;
      }
      if (kBwd) {
        float d = 0.0f;
        if (active) {
          const float4 hv = __ldcs(reinterpret_cast<const float4*>(f.S + off));
          d = val.x * hv.x + val.y * hv.y + val.z * hv.z + val.w * hv.w;
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
      const int c = p.nc - 1 - (k0 + k);
      float d = 0.0f;
      for (int w = 0; w < kSpThreads / 32; ++w) d += s_da[k][w];
      f.dapart[((size_t)bh * p.nc + c) * p.sp_neblk + eblk] = d;
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
