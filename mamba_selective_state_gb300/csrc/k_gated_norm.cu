// k_gated_norm.cu -- gated RMSNorm of the Mamba-2 block (the normalisation
// applied to the scan's output, gated by the block's z branch), forward and
// backward, and its C ABI (include/ssd.h).
//
// The operation is memory-bound: per element the forward reads y and z and
// writes out (6 bytes in bf16), the backward reads y, z and dout and writes
// dy and dz (10 bytes); everything else is a per-(row, group) sum of
// squares, a per-(row, group) projection and the column sums of dweight.
//
// Work split.  A (row, group) unit is handled by a team of nw warps in which
// every lane owns one 16-byte piece (8 bf16 or 4 fp32 values) of the group:
// nw = ceil(pieces per group / 32).  Each tensor is read exactly once with
// 128-bit streaming loads and written once with 128-bit streaming stores;
// the group sums are warp shuffles, plus one shared-memory exchange across
// the team's warps (named barrier per team) when nw > 1.  A CTA holds as many
// whole teams as fit in 256 threads (512 for nw > 8), and the grid is sized
// to the CTAs the device keeps resident at once (SM count x occupancy).
//
// Backward teams are persistent and own a fixed column group and a fixed
// slice of rows (team (s, k): group k, rows s, s + S, s + 2S, ...), keeping
// the group's dweight partial sums in registers and loading
// the next row's inputs while the current row is processed.  Each team
// writes its partial dweight to the workspace ((S, dim) fp32); a second
// kernel folds the S partials of every column in a fixed order (page "Cake
// RMSNorm", flashinfer PR 6997, section "Fixed-order tree fold reduction"),
// so dweight does not depend on scheduling.  The pages' bulk-copy
// producer/consumer pipeline for the norm backward is not needed here: no
// byte is reused across rows, and register double-buffering already keeps
// each SM's loads in flight.
#include <string.h>

#include "ssd_internal.cuh"

namespace ssd {

// ssd_api.cu: SSD_OK on an sm_103 device, else SSD_ERR_UNSUPPORTED (or SSD_ERR_CUDA).
int device_check();

namespace {

constexpr int kMaxTeamWarps = 16;   // pieces per group <= 512
constexpr int kMaxSlices = 1024;    // row slices of the backward (bounds the workspace)

struct NormArgs {
  const void* y;
  const void* z;
  const float* w;
  void* out;
  float* rstd;
  const void* dout;
  void* dy;
  void* dz;
  float* part;  // (S, dim) fp32 dweight partials
  long long rows;
  int dim, gs, G, npc, nw, tpc, S;
  float inv_gs, eps;
};

template <typename T>
struct Piece;
template <>
struct Piece<float> {
  static constexpr int n = 4;
  static __device__ __forceinline__ void unpack(const uint4& u, float* v) {
    v[0] = __uint_as_float(u.x); v[1] = __uint_as_float(u.y);
    v[2] = __uint_as_float(u.z); v[3] = __uint_as_float(u.w);
  }
  static __device__ __forceinline__ uint4 pack(const float* v) {
    return make_uint4(__float_as_uint(v[0]), __float_as_uint(v[1]), __float_as_uint(v[2]),
                      __float_as_uint(v[3]));
  }
};
template <>
struct Piece<__nv_bfloat16> {
  static constexpr int n = 8;
  static __device__ __forceinline__ void unpack2(uint32_t w, float* v) {
    v[0] = __uint_as_float(w << 16);           // element at the lower address
    v[1] = __uint_as_float(w & 0xffff0000u);
  }
  static __device__ __forceinline__ void unpack(const uint4& u, float* v) {
    unpack2(u.x, v); unpack2(u.y, v + 2); unpack2(u.z, v + 4); unpack2(u.w, v + 6);
  }
  static __device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
  }
  static __device__ __forceinline__ uint4 pack(const float* v) {
    return make_uint4(pack2(v[0], v[1]), pack2(v[2], v[3]), pack2(v[4], v[5]), pack2(v[6], v[7]));
  }
};

// Logistic function with the fast exponential and division.  The exponent
// is capped at 80 so that 1 + e stays finite and below 2^126, the range in
// which the fast division is exact to a few ulp; for z < -80 this returns
// about 1.8e-35 instead of e^z, far below any tolerance.
__device__ __forceinline__ float sigmoid_fast(float z) {
  return __fdividef(1.0f, 1.0f + __expf(fminf(-z, 80.0f)));
}

__device__ __forceinline__ float warp_allsum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;  // IEEE addition commutes, so every lane holds the same bits
}

__device__ __forceinline__ void team_barrier(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Sum over the lanes of a team of nw warps; every lane gets the same value.
// red: nw floats of shared memory owned by the team; barrier id 1 + team.
__device__ __forceinline__ float team_sum(float v, int nw, int team, int wi, int lane, float* red) {
  v = warp_allsum(v);
  if (nw == 1) return v;
  if (lane == 0) red[wi] = v;
  team_barrier(1 + team, nw * 32);
  float s = 0.0f;
  for (int i = 0; i < nw; ++i) s += red[i];  // fixed order
  team_barrier(1 + team, nw * 32);           // red is rewritten by the next sum
  return s;
}

// g = y * silu(z) (or y) for the values of one piece, from the raw pieces of
// y and z and sigmoid(z).
template <typename T, bool kGate>
__device__ __forceinline__ void gated_values(const uint4& yr, const uint4& zr, const float* sg,
                                             float* g) {
  constexpr int V = Piece<T>::n;
  Piece<T>::unpack(yr, g);
  if (kGate) {
    float zv[V];
    Piece<T>::unpack(zr, zv);
#pragma unroll
    for (int i = 0; i < V; ++i) g[i] *= zv[i] * sg[i];
  }
}

template <typename T, bool kGate, int kThreads>
__global__ void __launch_bounds__(kThreads) gated_norm_fwd_kernel(NormArgs a) {
  constexpr int V = Piece<T>::n;
  __shared__ float red[kThreads / 32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int team = warp / a.nw, wi = warp - team * a.nw;
  const int tl = wi * 32 + lane;  // lane within the team = piece index in the group
  const bool has_piece = tl < a.npc;
  float* tred = red + team * a.nw;
  const long long nunits = a.rows * a.G;
  const long long stride = (long long)gridDim.x * a.tpc;
  for (long long u = (long long)blockIdx.x * a.tpc + team; u < nunits; u += stride) {
    const long long r = u / a.G;
    const int k = (int)(u - r * a.G);
    const int col = k * a.gs + tl * V;
    const long long off = r * a.dim + col;
    float g[V];
    float ss = 0.0f;
    if (has_piece) {
      Piece<T>::unpack(__ldcs(reinterpret_cast<const uint4*>(static_cast<const T*>(a.y) + off)), g);
      if (kGate) {
        float zv[V];
        Piece<T>::unpack(__ldcs(reinterpret_cast<const uint4*>(static_cast<const T*>(a.z) + off)), zv);
#pragma unroll
        for (int i = 0; i < V; ++i) g[i] *= zv[i] * sigmoid_fast(zv[i]);
      }
#pragma unroll
      for (int i = 0; i < V; ++i) ss = fmaf(g[i], g[i], ss);
    }
    const float rstd = rsqrtf(team_sum(ss, a.nw, team, wi, lane, tred) * a.inv_gs + a.eps);
    if (has_piece) {
      float wv[V];
#pragma unroll
      for (int i = 0; i < V; i += 4) {
        const float4 q = __ldg(reinterpret_cast<const float4*>(a.w + col + i));
        wv[i] = q.x; wv[i + 1] = q.y; wv[i + 2] = q.z; wv[i + 3] = q.w;
      }
#pragma unroll
      for (int i = 0; i < V; ++i) g[i] = (g[i] * rstd) * wv[i];
      __stcs(reinterpret_cast<uint4*>(static_cast<T*>(a.out) + off), Piece<T>::pack(g));
    }
    if (a.rstd != nullptr && tl == 0) a.rstd[u] = rstd;
  }
}

template <typename T, bool kGate, int kThreads>
__global__ void __launch_bounds__(kThreads, 768 / kThreads) gated_norm_bwd_kernel(NormArgs a) {
  constexpr int V = Piece<T>::n;
  __shared__ float red[kThreads / 32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int team = warp / a.nw, wi = warp - team * a.nw;
  const long long t = (long long)blockIdx.x * a.tpc + team;  // global team id
  if (t >= (long long)a.S * a.G) return;                     // whole teams leave together
  const int k = (int)(t % a.G), s = (int)(t / a.G);
  const int tl = wi * 32 + lane;
  const bool has_piece = tl < a.npc;
  float* tred = red + team * a.nw;
  const int col = k * a.gs + tl * V;
  const T* yb = static_cast<const T*>(a.y) + col;
  const T* zb = kGate ? static_cast<const T*>(a.z) + col : nullptr;
  const T* db = static_cast<const T*>(a.dout) + col;

  float dw[V];
#pragma unroll
  for (int i = 0; i < V; ++i) dw[i] = 0.0f;
  const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
  uint4 yr = zero, zr = zero, dr = zero;
  if (has_piece && s < a.rows) {
    const long long off = (long long)s * a.dim;
    yr = __ldcs(reinterpret_cast<const uint4*>(yb + off));
    if (kGate) zr = __ldcs(reinterpret_cast<const uint4*>(zb + off));
    dr = __ldcs(reinterpret_cast<const uint4*>(db + off));
  }
  for (long long r = s; r < a.rows; r += a.S) {
    // inputs of this team's next row, loaded while this row is processed
    const long long rn = r + a.S;
    uint4 yn = zero, zn = zero, dn = zero;
    if (has_piece && rn < a.rows) {
      const long long off = rn * a.dim;
      yn = __ldcs(reinterpret_cast<const uint4*>(yb + off));
      if (kGate) zn = __ldcs(reinterpret_cast<const uint4*>(zb + off));
      dn = __ldcs(reinterpret_cast<const uint4*>(db + off));
    }
    // sigmoid(z) is kept for the row; g = y * silu(z) is recomputed from the
    // raw pieces in each pass (bitwise the same each time), which keeps the
    // kernel within the registers of three CTAs per SM
    float sg[V];
    float ss = 0.0f;
    {
      if (kGate) {
        float zv[V];
        Piece<T>::unpack(zr, zv);
#pragma unroll
        for (int i = 0; i < V; ++i) sg[i] = sigmoid_fast(zv[i]);
      }
      float g[V];
      gated_values<T, kGate>(yr, zr, sg, g);
#pragma unroll
      for (int i = 0; i < V; ++i) ss = fmaf(g[i], g[i], ss);
    }
    // lanes without a piece hold zeros and add nothing to either sum
    const float rstd = rsqrtf(team_sum(ss, a.nw, team, wi, lane, tred) * a.inv_gs + a.eps);
    // the team's weights are re-read from L1 every row rather than held in
    // registers (they are the same few hundred bytes for every row)
    float wv[V];
#pragma unroll
    for (int i = 0; i < V; ++i) wv[i] = 0.0f;
    if (has_piece) {
#pragma unroll
      for (int i = 0; i < V; i += 4) {
        const float4 q = __ldg(reinterpret_cast<const float4*>(a.w + col + i));
        wv[i] = q.x; wv[i + 1] = q.y; wv[i + 2] = q.z; wv[i + 3] = q.w;
      }
    }
    float sdn = 0.0f;
    {
      float g[V], dov[V];
      gated_values<T, kGate>(yr, zr, sg, g);
      Piece<T>::unpack(dr, dov);
#pragma unroll
      for (int i = 0; i < V; ++i) sdn = fmaf(dov[i] * wv[i], g[i] * rstd, sdn);
    }
    const float c = team_sum(sdn, a.nw, team, wi, lane, tred) * a.inv_gs;
    if (has_piece) {
      const long long off = r * a.dim;
      float g[V], dov[V], dyv[V];
      gated_values<T, kGate>(yr, zr, sg, g);
      Piece<T>::unpack(dr, dov);
      if (kGate) {
        float yv[V], zv[V], dzv[V];
        Piece<T>::unpack(yr, yv);
        Piece<T>::unpack(zr, zv);
#pragma unroll
        for (int i = 0; i < V; ++i) {
          const float n = g[i] * rstd;
          const float dg = rstd * (dov[i] * wv[i] - n * c);
          dw[i] = fmaf(dov[i], n, dw[i]);
          dyv[i] = dg * (zv[i] * sg[i]);
          dzv[i] = dg * yv[i] * sg[i] * (1.0f + zv[i] * (1.0f - sg[i]));
        }
        __stcs(reinterpret_cast<uint4*>(static_cast<T*>(a.dz) + col + off), Piece<T>::pack(dzv));
      } else {
#pragma unroll
        for (int i = 0; i < V; ++i) {
          const float n = g[i] * rstd;
          dw[i] = fmaf(dov[i], n, dw[i]);
          dyv[i] = rstd * (dov[i] * wv[i] - n * c);
        }
      }
      __stcs(reinterpret_cast<uint4*>(static_cast<T*>(a.dy) + col + off), Piece<T>::pack(dyv));
    }
    yr = yn; zr = zn; dr = dn;
  }
  if (has_piece) {
    float* pp = a.part + (long long)s * a.dim + col;
#pragma unroll
    for (int i = 0; i < V; i += 4)
      *reinterpret_cast<float4*>(pp + i) = make_float4(dw[i], dw[i + 1], dw[i + 2], dw[i + 3]);
  }
}

// dweight[j] = sum over the S slices of part[s][j], in a fixed order: thread
// (column c, lane q) of a CTA adds slices q, q + 8, q + 16, ... in turn, then
// the eight lane sums of a column are folded as a binary tree.
constexpr int kFoldCols = 32, kFoldLanes = 8;
__global__ void __launch_bounds__(kFoldCols * kFoldLanes)
    gated_norm_dw_fold_kernel(const float* __restrict__ part, int S, int dim, float* __restrict__ dw) {
  __shared__ float acc[kFoldLanes][kFoldCols];
  const int cx = threadIdx.x % kFoldCols, q = threadIdx.x / kFoldCols;
  const int j = blockIdx.x * kFoldCols + cx;
  float v = 0.0f;
  if (j < dim)
    for (int s = q; s < S; s += kFoldLanes) v += part[(long long)s * dim + j];
  acc[q][cx] = v;
  __syncthreads();
  if (q == 0 && j < dim) {
    const float a01 = acc[0][cx] + acc[1][cx], a23 = acc[2][cx] + acc[3][cx];
    const float a45 = acc[4][cx] + acc[5][cx], a67 = acc[6][cx] + acc[7][cx];
    dw[j] = (a01 + a23) + (a45 + a67);
  }
}

struct NormPlan {
  long long rows;
  int dim, gs, G, npc, nw, tpc, threads, S_max;
  int dtype, flags;
  float eps;
  size_t ws_bytes;
};

int make_norm_plan(const ssd_norm_problem* pr, NormPlan* p) {
  if (!pr) return SSD_ERR_INVALID_ARGUMENT;
  if (pr->rows < 1 || pr->dim < 1 || pr->group_size < 1) return SSD_ERR_INVALID_ARGUMENT;
  if (pr->dim % pr->group_size != 0) return SSD_ERR_INVALID_ARGUMENT;
  if (pr->dtype != SSD_F32 && pr->dtype != SSD_BF16) return SSD_ERR_INVALID_ARGUMENT;
  if (pr->flags & ~SSD_NORM_HAS_Z) return SSD_ERR_INVALID_ARGUMENT;
  if (!(pr->eps >= 0.0f) || pr->eps > 3.0e38f) return SSD_ERR_INVALID_ARGUMENT;  // also rejects NaN
  const int V = pr->dtype == SSD_BF16 ? 8 : 4;
  if (pr->group_size % V != 0) return SSD_ERR_UNSUPPORTED;
  const long long npc = pr->group_size / V;
  if (npc > 32LL * kMaxTeamWarps) return SSD_ERR_UNSUPPORTED;
  // 32-bit column indices; at most 2^40 elements per tensor
  if (pr->dim > (1LL << 30) || pr->rows > (1LL << 40) / pr->dim) return SSD_ERR_UNSUPPORTED;
  p->rows = pr->rows;
  p->dim = (int)pr->dim;
  p->gs = (int)pr->group_size;
  p->G = (int)(pr->dim / pr->group_size);
  p->npc = (int)npc;
  p->nw = (int)((npc + 31) / 32);
  const int cta_warps = p->nw <= 8 ? 8 : 16;
  p->tpc = cta_warps / p->nw;
  p->threads = p->tpc * p->nw * 32;
  p->dtype = pr->dtype;
  p->flags = pr->flags;
  p->eps = pr->eps;
  // slices of the backward: at most one per row, at most kMaxSlices, and
  // at least one per group
  p->S_max = (int)(pr->rows < kMaxSlices ? pr->rows : kMaxSlices);
  p->ws_bytes = (size_t)p->S_max * (size_t)p->dim * sizeof(float);
  return SSD_OK;
}

bool misaligned16(const void* ptr) { return ptr && (reinterpret_cast<uintptr_t>(ptr) & 15u); }

NormArgs base_args(const NormPlan& p) {
  NormArgs a;
  memset(&a, 0, sizeof(a));
  a.rows = p.rows;
  a.dim = p.dim;
  a.gs = p.gs;
  a.G = p.G;
  a.npc = p.npc;
  a.nw = p.nw;
  a.tpc = p.tpc;
  a.inv_gs = 1.0f / (float)p.gs;
  a.eps = p.eps;
  return a;
}

template <typename T, bool kGate, int kThreads>
cudaError_t launch_fwd_t(const NormPlan& p, const NormArgs& a, cudaStream_t s) {
  auto kern = gated_norm_fwd_kernel<T, kGate, kThreads>;
  int occ = 0;
  cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, p.threads, 0);
  if (e != cudaSuccess) return e;
  if (occ < 1) occ = 1;
  const long long units = p.rows * p.G;
  long long grid = (units + p.tpc - 1) / p.tpc;
  const long long cap = (long long)device_sm_count() * occ;
  if (grid > cap) grid = cap;
  set_kernel_name("gated_norm_fwd");
  kern<<<(unsigned)grid, p.threads, 0, s>>>(a);
  return cudaGetLastError();
}

template <typename T, bool kGate, int kThreads>
cudaError_t launch_bwd_t(const NormPlan& p, NormArgs& a, cudaStream_t s) {
  auto kern = gated_norm_bwd_kernel<T, kGate, kThreads>;
  int occ = 0;
  cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, p.threads, 0);
  if (e != cudaSuccess) return e;
  if (occ < 1) occ = 1;
  // as many slices as keep every resident team busy, within [1, S_max]
  const long long teams = (long long)device_sm_count() * occ * p.tpc;
  long long S = teams / p.G;
  if (S > p.S_max) S = p.S_max;
  if (S < 1) S = 1;
  a.S = (int)S;
  const long long grid = (S * p.G + p.tpc - 1) / p.tpc;
  set_kernel_name("gated_norm_bwd");
  kern<<<(unsigned)grid, p.threads, 0, s>>>(a);
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_fwd_dtype(const NormPlan& p, const NormArgs& a, cudaStream_t s) {
  const bool gate = (p.flags & SSD_NORM_HAS_Z) != 0;
  if (p.threads <= 256)
    return gate ? launch_fwd_t<T, true, 256>(p, a, s) : launch_fwd_t<T, false, 256>(p, a, s);
  return gate ? launch_fwd_t<T, true, 512>(p, a, s) : launch_fwd_t<T, false, 512>(p, a, s);
}

template <typename T>
cudaError_t launch_bwd_dtype(const NormPlan& p, NormArgs& a, cudaStream_t s) {
  const bool gate = (p.flags & SSD_NORM_HAS_Z) != 0;
  if (p.threads <= 256)
    return gate ? launch_bwd_t<T, true, 256>(p, a, s) : launch_bwd_t<T, false, 256>(p, a, s);
  return gate ? launch_bwd_t<T, true, 512>(p, a, s) : launch_bwd_t<T, false, 512>(p, a, s);
}

#define NORM_LAUNCH(expr)                       \
  do {                                          \
    prof_before(s);                             \
    cudaError_t e_ = (expr);                    \
    prof_after(s);                              \
    if (e_ != cudaSuccess) return SSD_ERR_CUDA; \
  } while (0)

}  // namespace

}  // namespace ssd

using namespace ssd;

extern "C" {

int ssd_gated_rmsnorm_fwd(const ssd_norm_problem* prob, const void* y, const void* z,
                          const float* weight, void* out, float* rstd, ssd_stream_t stream) {
  NormPlan p;
  int rc = make_norm_plan(prob, &p);
  if (rc != SSD_OK) return rc;
  if (!y || !weight || !out) return SSD_ERR_INVALID_ARGUMENT;
  if (((p.flags & SSD_NORM_HAS_Z) != 0) != (z != nullptr)) return SSD_ERR_INVALID_ARGUMENT;
  const void* ptrs[] = {y, z, weight, out, rstd};
  for (const void* q : ptrs)
    if (misaligned16(q)) return SSD_ERR_INVALID_ARGUMENT;
  rc = device_check();
  if (rc != SSD_OK) return rc;
  NormArgs a = base_args(p);
  a.y = y; a.z = z; a.w = weight; a.out = out; a.rstd = rstd;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (p.dtype == SSD_BF16)
    NORM_LAUNCH(launch_fwd_dtype<__nv_bfloat16>(p, a, s));
  else
    NORM_LAUNCH(launch_fwd_dtype<float>(p, a, s));
  return SSD_OK;
}

size_t ssd_gated_rmsnorm_bwd_workspace_bytes(const ssd_norm_problem* prob) {
  NormPlan p;
  return make_norm_plan(prob, &p) == SSD_OK ? p.ws_bytes : 0;
}

int ssd_gated_rmsnorm_bwd(const ssd_norm_problem* prob, const void* y, const void* z,
                          const float* weight, const void* dout, void* dy, void* dz,
                          float* dweight, void* workspace, size_t workspace_bytes,
                          ssd_stream_t stream) {
  NormPlan p;
  int rc = make_norm_plan(prob, &p);
  if (rc != SSD_OK) return rc;
  if (!y || !weight || !dout || !dy || !dweight || !workspace) return SSD_ERR_INVALID_ARGUMENT;
  const bool gate = (p.flags & SSD_NORM_HAS_Z) != 0;
  if (gate != (z != nullptr) || gate != (dz != nullptr)) return SSD_ERR_INVALID_ARGUMENT;
  const void* ptrs[] = {y, z, weight, dout, dy, dz, dweight, workspace};
  for (const void* q : ptrs)
    if (misaligned16(q)) return SSD_ERR_INVALID_ARGUMENT;
  if (workspace_bytes < p.ws_bytes) return SSD_ERR_WORKSPACE_TOO_SMALL;
  rc = device_check();
  if (rc != SSD_OK) return rc;
  NormArgs a = base_args(p);
  a.y = y; a.z = z; a.w = weight; a.dout = dout; a.dy = dy; a.dz = dz;
  a.part = static_cast<float*>(workspace);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (p.dtype == SSD_BF16)
    NORM_LAUNCH(launch_bwd_dtype<__nv_bfloat16>(p, a, s));
  else
    NORM_LAUNCH(launch_bwd_dtype<float>(p, a, s));
  // a.S now holds the slice count the backward kernel used
  set_kernel_name("gated_norm_dw_fold");
  NORM_LAUNCH((gated_norm_dw_fold_kernel<<<(p.dim + kFoldCols - 1) / kFoldCols,
                                           kFoldCols * kFoldLanes, 0, s>>>(
                   a.part, a.S, p.dim, dweight),
               cudaGetLastError()));
  return SSD_OK;
}

}  // extern "C"
