// k_dt.cu -- the per-token dt kernels of the SSD layer.
//
//  dt_cumsum (forward, step 1): dt_eff = softplus(dt + dt_bias_h) and the
//    chunk-local inclusive cumsum l_i = sum_{k<=i} dt_eff_k A_h, one warp per
//    (row, chunk, head) with an in-warp shuffle scan; also the chunk decay
//    a_c = exp(l_last) (0 when a sequence starts inside the chunk), and the
//    zeroing of the scan flags/tickets and the status word of this call.
//  dt_bwd (backward, last step): d(dt_eff A) = reverse cumsum of dL/dl inside
//    the chunk, then ddt = (ddt_eff + A_h d(dA)) * sigmoid(dt + dt_bias_h) and
//    per-chunk partials of dA and ddt_bias.
//  param_reduce: dA, dD, ddt_bias folded over (row, chunk[, token block]) in a
//    fixed order (one CTA per head, fixed-shape tree), so that the results are
//    bitwise reproducible (the fixed-order tree fold of page "flashinfer PR
//    6997 Cake RMSNorm" (blog.secrett2633.cloud), section "Fixed-order Tree
//    Fold Reduction").
#include "ssd_internal.cuh"

namespace ssd {

namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr int kHeadsPerCta = 8;  // one warp per head
constexpr int kMaxPerLane = 8;   // chunk <= 256 tokens

__device__ __forceinline__ float softplus_f(float z) {
  return fmaxf(z, 0.0f) + log1pf(expf(-fabsf(z)));
}
__device__ __forceinline__ float sigmoid_f(float z) {
  return z >= 0.0f ? 1.0f / (1.0f + expf(-z)) : expf(z) / (1.0f + expf(z));
}

template <typename T>
__global__ void __launch_bounds__(256) dt_cumsum_kernel(Plan p, Bufs f) {
  // Zero this call's scan flags and tickets and the status word.
  {
    const long long nflags = (long long)p.sp_chains * p.sp_nslot;
    const long long nthr = (long long)gridDim.x * gridDim.y * gridDim.z * blockDim.x;
    long long gid = (((long long)blockIdx.z * gridDim.y + blockIdx.y) * gridDim.x + blockIdx.x) *
                        blockDim.x + threadIdx.x;
    for (long long i = gid; i < nflags; i += nthr) {
      f.flags_fwd[i] = 0;
      f.flags_bwd[i] = 0;
    }
    if (gid == 0) {
      f.hdr->status = 0;
      f.hdr->ticket_fwd = 0;
      f.hdr->ticket_bwd = 0;
      if (p.kept_mode == 1) f.hdr->kept_sig = p.kept_sig_write;
    }
  }
  const int c = blockIdx.x, bi = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.z * kHeadsPerCta + warp;
  if (h >= p.H) return;
  const int t0 = c * p.Q;
  const int len = min(p.Q, p.L - t0);
  const int R = (p.Q + 31) >> 5;
  const float bias = f.dt_bias[h], Ah = f.A[h];
  const T* dt = static_cast<const T*>(f.dt);
  float de[kMaxPerLane], lv[kMaxPerLane];
  float run = 0.0f;
#pragma unroll
  for (int k = 0; k < kMaxPerLane; ++k) {
    float v = 0.0f;
    const int i = lane * R + k;
    if (k < R && i < len) v = softplus_f(to_f(dt[((long long)bi * p.L + t0 + i) * p.H + h]) + bias);
    de[k] = v;
    run += v * Ah;
    lv[k] = run;
  }
  // in-warp inclusive scan of the lane totals (log-step, one lane per span)
  float s = run;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const float o = __shfl_up_sync(kFull, s, d);
    if (lane >= d) s += o;
  }
  float excl = __shfl_up_sync(kFull, s, 1);
  if (lane == 0) excl = 0.0f;
  const long long base = ((long long)bi * p.H + h) * p.Lp + t0;
#pragma unroll
  for (int k = 0; k < kMaxPerLane; ++k) {
    const int i = lane * R + k;
    if (k < R && i < p.Q) {
      f.dte[base + i] = de[k];
      f.lcs[base + i] = excl + lv[k];
    }
  }
  const float l_last = __shfl_sync(kFull, s, 31);
  if (lane == 0) {
    float a = expf(l_last);
    if (f.seq != nullptr && seg_of(p, f, bi, (long long)t0 + len - 1) != seg_in_of(p, f, bi, c))
      a = 0.0f;
    f.achunk[((long long)bi * p.H + h) * p.nc + c] = a;
  }
}

template <typename T>
__global__ void __launch_bounds__(256) dt_bwd_kernel(Plan p, Bufs f) {
  const int c = blockIdx.x, bi = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.z * kHeadsPerCta + warp;
  if (h >= p.H) return;
  const int t0 = c * p.Q;
  const int len = min(p.Q, p.L - t0);
  const int R = (p.Q + 31) >> 5;
  const long long bh = (long long)bi * p.H + h;
  const long long base = bh * p.Lp + t0;
  // extra gradient of the last token's cumsum: the chunk-state weights'
  // dependence on l_last (summed over token blocks) and the chunk decay a_c
  float extra = 0.0f;
  if (lane == 0) {
    const float* u = f.udu + (bh * p.nc + c) * p.cb_ntb;
    for (int tb = 0; tb < p.cb_ntb; ++tb) extra += u[tb];
    const float a = f.achunk[bh * p.nc + c];
    if (a != 0.0f) {
      float da = 0.0f;
      const float* dp = f.dapart + (bh * p.nc + c) * p.da_stride;
      for (int k = 0; k < p.da_nsum; ++k) da += dp[k];
      extra += a * da;
    }
  }
  extra = __shfl_sync(kFull, extra, 0);
  float dl[kMaxPerLane];
  float tot = 0.0f;
#pragma unroll
  for (int k = 0; k < kMaxPerLane; ++k) {
    const int i = lane * R + k;
    float v = 0.0f;
    if (k < R && i < len) v = f.dl[base + i] + (i == len - 1 ? extra : 0.0f);
    dl[k] = v;
    tot += v;
  }
  // suffix sums across lanes: lanes to the right hold later tokens
  float s = tot;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const float o = __shfl_down_sync(kFull, s, d);
    if (lane + d < 32) s += o;
  }
  float after = __shfl_down_sync(kFull, s, 1);  // sum over lanes > lane
  if (lane == 31) after = 0.0f;
  const float bias = f.dt_bias[h], Ah = f.A[h];
  const T* dt = static_cast<const T*>(f.dt);
  T* ddt = static_cast<T*>(f.ddt);
  float pA = 0.0f, pb = 0.0f;
  float run = after;
#pragma unroll
  for (int k = kMaxPerLane - 1; k >= 0; --k) {
    const int i = lane * R + k;
    if (k < R && i < len) {
      run += dl[k];  // d(dA_i) = sum_{i' >= i} dl_i'
      const float de = f.dte[base + i];
      const float g = f.ddte[base + i] + Ah * run;
      const long long ti = ((long long)bi * p.L + t0 + i) * p.H + h;
      const float v = g * sigmoid_f(to_f(dt[ti]) + bias);
      ddt[ti] = from_f<T>(v);
      pA += de * run;
      pb += v;
    }
  }
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) {
    pA += __shfl_xor_sync(kFull, pA, d);
    pb += __shfl_xor_sync(kFull, pb, d);
  }
  if (lane == 0) {
    f.pdA[((long long)bi * p.nc + c) * p.H + h] = pA;
    f.pdb[((long long)bi * p.nc + c) * p.H + h] = pb;
  }
}

__device__ float block_sum_fixed(float v, float* sm) {
  // fixed-shape tree over 256 threads: deterministic for a fixed input order
  sm[threadIdx.x] = v;
  __syncthreads();
  for (int s = 128; s > 0; s >>= 1) {
    if (threadIdx.x < s) sm[threadIdx.x] += sm[threadIdx.x + s];
    __syncthreads();
  }
  const float r = sm[0];
  __syncthreads();
  return r;
}

__global__ void __launch_bounds__(256) param_reduce_kernel(Plan p, Bufs f) {
  __shared__ float sm[256];
  const int h = blockIdx.x;
  const long long n1 = (long long)p.b * p.nc;
  const long long n2 = n1 * p.cb_ntb;
  float a = 0.0f, b = 0.0f, d = 0.0f;
  for (long long k = threadIdx.x; k < n1; k += 256) {
    a += f.pdA[k * p.H + h];
    b += f.pdb[k * p.H + h];
  }
  for (long long k = threadIdx.x; k < n2; k += 256) d += f.pdD[k * p.H + h];
  a = block_sum_fixed(a, sm);
  b = block_sum_fixed(b, sm);
  d = block_sum_fixed(d, sm);
  if (threadIdx.x == 0) {
    f.dA[h] = a;
    f.ddt_bias[h] = b;
    f.dD[h] = d;
  }
}

// Clears the status word of a call whose kernels do not (the single-pass
// forward).  A kernel on the call's stream rather than a memset: a memset can
// be served by a copy engine and queue behind the caller's host copies.
// It also writes the kept-intermediates stamp (mode 1) or checks it (mode 2).
__global__ void status_reset_kernel(WsHeader* hdr, int mode, int sig, int sig_write) {
  int st = 0;
  if (mode == 1) hdr->kept_sig = sig_write;
  if (mode == 2 && (hdr->kept_sig & ~kKeptF32) != sig) st = kDevNoKept;
  hdr->status = st;
}

__global__ void __launch_bounds__(256) kept_scan_reset_kernel(Plan p, Bufs f) {
  const long long nflags = (long long)p.sp_chains * p.sp_nslot;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < nflags;
       i += (long long)gridDim.x * blockDim.x)
    f.flags_bwd[i] = 0;
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    f.hdr->ticket_bwd = 0;
    f.hdr->status = f.hdr->kept_sig == (p.kept_sig | kKeptF32) ? 0 : kDevNoKept;
  }
}

}  // namespace

cudaError_t launch_status_reset(const Plan& p, const Bufs& f, cudaStream_t s) {
  set_kernel_name("status_reset");
  status_reset_kernel<<<1, 1, 0, s>>>(f.hdr, p.kept_mode, p.kept_sig, p.kept_sig_write);
  return cudaGetLastError();
}

cudaError_t launch_kept_scan_reset(const Plan& p, const Bufs& f, cudaStream_t s) {
  set_kernel_name("kept_scan_reset");
  const long long nflags = (long long)p.sp_chains * p.sp_nslot;
  const long long blocks = (nflags + 255) / 256;
  const int grid = (int)(blocks < 1 ? 1 : (blocks > 1024 ? 1024 : blocks));
  kept_scan_reset_kernel<<<grid, 256, 0, s>>>(p, f);
  return cudaGetLastError();
}

cudaError_t launch_dt_cumsum(const Plan& p, const Bufs& f, cudaStream_t s) {
  set_kernel_name("dt_cumsum");
  dim3 grid(p.nc, p.b, (p.H + kHeadsPerCta - 1) / kHeadsPerCta);
  if (p.dtype == SSD_BF16)
    dt_cumsum_kernel<__nv_bfloat16><<<grid, 256, 0, s>>>(p, f);
  else
    dt_cumsum_kernel<float><<<grid, 256, 0, s>>>(p, f);
  return cudaGetLastError();
}

cudaError_t launch_dt_bwd(const Plan& p, const Bufs& f, cudaStream_t s) {
  set_kernel_name("dt_bwd");
  dim3 grid(p.nc, p.b, (p.H + kHeadsPerCta - 1) / kHeadsPerCta);
  if (p.dtype == SSD_BF16)
    dt_bwd_kernel<__nv_bfloat16><<<grid, 256, 0, s>>>(p, f);
  else
    dt_bwd_kernel<float><<<grid, 256, 0, s>>>(p, f);
  return cudaGetLastError();
}

cudaError_t launch_param_reduce(const Plan& p, const Bufs& f, cudaStream_t s) {
  set_kernel_name("param_reduce");
  param_reduce_kernel<<<p.H, 256, 0, s>>>(p, f);
  return cudaGetLastError();
}

}  // namespace ssd
