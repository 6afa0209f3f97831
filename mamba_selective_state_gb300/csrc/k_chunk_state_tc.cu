// k_chunk_state_tc.cu -- chunk states on the 5th-generation tensor cores.
//
//   chunk_state : S_c[n][p]   = sum_j sv_j exp(l_last - l_j) dt_eff_j  B_j[n] x_j[p]
//   chunk_dstate: dHloc[n][p] = sum_i cv_i exp(l_i) C_i[n] dy_i[p]
// (page "llm-mamba-200" (gigipick.blogspot.com), section 3: the carry-out
// state of each chunk; the backward's carry gradient has the same shape).
//
// One CTA computes the chunk states of two heads h, h+1 of the same group:
// a tcgen05.mma with M = 128 = 2 heads x headdim 64 (A = the two x tiles,
// token-weighted, MN-major), N = d_state (B tile of the group, MN-major) and
// K = the chunk's tokens, accumulated in fp32 in tensor memory.  Tokens are
// streamed in stages of 32 by TMA (128-byte swizzle) through a two-stage
// mbarrier pipeline; the per-token weights are applied to the x rows in
// shared memory before the MMA reads them.  The epilogue reads the
// accumulator back with tcgen05.ld and writes S in the (d_state, headdim)
// layout, one coalesced 128-byte row per warp and state index.
#include "ssd_internal.cuh"
#include "tc_common.cuh"
#include "tma_host.h"

namespace ssd {

namespace {

using namespace tc;

constexpr int kStageTok = 32;   // tokens per pipeline stage (small stages: four CTAs per SM)
constexpr int kThr = 128;       // 4 warps: one per TMEM lane quadrant
constexpr uint32_t kABytes = 2 * kStageTok * 128;  // two heads x kStageTok tokens x 64 bf16

__host__ __device__ inline uint32_t round1024(uint32_t v) { return (v + 1023u) & ~1023u; }

struct StateGeom {
  int bw;          // bytes per B row in one box (2 * min(N, 64))
  int nbox;        // boxes along d_state
  uint32_t box;    // bytes of one B box (kStageTok tokens)
  uint32_t stage;  // bytes of one stage (A + B), 1024-aligned
  uint32_t swz;    // descriptor swizzle code of B
  uint32_t ncols;  // TMEM columns
};

__host__ __device__ inline StateGeom state_geom(int N) {
  StateGeom g;
  g.bw = 2 * (N < 64 ? N : 64);
  g.nbox = N >= 64 ? N / 64 : 1;
  g.box = (uint32_t)kStageTok * g.bw;
  g.stage = round1024(kABytes + g.nbox * g.box);
  g.swz = g.bw == 128 ? kSwz128 : (g.bw == 64 ? kSwz64 : kSwz32);
  g.ncols = N < 32 ? 32 : N;
  return g;
}

__device__ __forceinline__ uint32_t scale_bf16x2(uint32_t v, float w) {
  __nv_bfloat162 h = *reinterpret_cast<__nv_bfloat162*>(&v);
  float2 f = __bfloat1622float2(h);
  __nv_bfloat162 r = __floats2bfloat162_rn(f.x * w, f.y * w);
  return *reinterpret_cast<uint32_t*>(&r);
}

template <bool kDstates>
__global__ void __launch_bounds__(kThr) chunk_state_tc_kernel(Plan p, Bufs f,
                                                               const __grid_constant__ CUtensorMap tmX,
                                                               const __grid_constant__ CUtensorMap tmB) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const StateGeom G = state_geom(p.N);
  const int c = blockIdx.x, h0 = 2 * blockIdx.y, bi = blockIdx.z;
  const int g = h0 / p.hpg;
  const int tid = threadIdx.x;
  const int t0 = c * p.Q, len = min(p.Q, p.L - t0);
  const int nkb = (len + kStageTok - 1) / kStageTok;
  float* w = reinterpret_cast<float*>(sm + 2 * G.stage);       // [2][Q]
  uint64_t* bar = reinterpret_cast<uint64_t*>(w + 2 * p.Q);     // full[2], done[2]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + 4);

  // token weights of both heads
  {
    const int s_ref = kDstates ? seg_in_of(p, f, bi, c) : seg_of(p, f, bi, (long long)t0 + len - 1);
    for (int idx = tid; idx < 2 * p.Q; idx += kThr) {
      const int hh = idx / p.Q, j = idx - hh * p.Q;
      const long long bh = (long long)bi * p.H + h0 + hh;
      const float* lc = f.lcs + bh * p.Lp + t0;
      float v = 0.0f;
      if (j < len && seg_of(p, f, bi, (long long)t0 + j) == s_ref)
        v = kDstates ? expf(lc[j]) : expf(lc[len - 1] - lc[j]) * f.dte[bh * p.Lp + t0 + j];
      w[idx] = v;
    }
  }
  if (tid == 0) {
    for (int i = 0; i < 4; ++i) mbar_init(&bar[i], 1);
    mbar_fence_init();
    prefetch_tmap(&tmX);
    prefetch_tmap(&tmB);
  }
  if (tid < 32) tmem_alloc(tmem_slot, G.ncols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t idesc = idesc_bf16(128, p.N, 1, 1);
  bool ok = true;

  auto issue = [&](int kb) {
    uint8_t* A = sm + (kb & 1) * G.stage;
    uint8_t* Bt = A + kABytes;
    const int tok = t0 + kb * kStageTok;
    mbar_expect_tx(&bar[kb & 1], kABytes + G.nbox * G.box);
    tma_load_4d(A, &tmX, &bar[kb & 1], 0, h0, tok, bi);
    tma_load_4d(A + kABytes / 2, &tmX, &bar[kb & 1], 0, h0 + 1, tok, bi);
    for (int q = 0; q < G.nbox; ++q) tma_load_4d(Bt + q * G.box, &tmB, &bar[kb & 1], q * 64, g, tok, bi);
  };
  if (tid == 0) {
    issue(0);
    if (nkb > 1) issue(1);
  }
  for (int kb = 0; kb < nkb; ++kb) {
    const int s = kb & 1;
    const uint32_t ph = (kb >> 1) & 1;
    uint8_t* A = sm + s * G.stage;
    uint8_t* Bt = A + kABytes;
    if (!mbar_wait(&bar[s], ph)) ok = false;
    {  // scale the stage's 2 x kStageTok x rows (128 bytes each) by their token weights
      constexpr int kRowsStage = 2 * kStageTok;
      constexpr int kPer = kRowsStage >= kThr ? 1 : kThr / kRowsStage;  // threads per row
      constexpr int kU4 = 8 / kPer;                                     // 16-byte pieces per thread
      const int row = tid / kPer, part = tid % kPer;
      const int hh = row / kStageTok, r = row % kStageTok;
      const float wv = w[hh * p.Q + kb * kStageTok + r];
      uint4* rp = reinterpret_cast<uint4*>(A + hh * (kABytes / 2) + r * 128) + part * kU4;
#pragma unroll
      for (int q = 0; q < kU4; ++q) {
        uint4 v = rp[q];
        v.x = scale_bf16x2(v.x, wv);
        v.y = scale_bf16x2(v.y, wv);
        v.z = scale_bf16x2(v.z, wv);
        v.w = scale_bf16x2(v.w, wv);
        rp[q] = v;
      }
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    if (tid == 0) {
      tc_fence_after();
#pragma unroll
      for (int ks = 0; ks < kStageTok / 16; ++ks) {
        const uint64_t da = smem_desc(smem_u32(A) + ks * 16 * 128, kABytes / 2, 1024, kSwz128);
        const uint64_t db = smem_desc(smem_u32(Bt) + ks * 16 * G.bw, G.box, 8 * G.bw, G.swz);
        mma_bf16(tmem, da, db, idesc, (kb | ks) != 0);
      }
      mma_commit(&bar[2 + s]);
      if (kb + 2 < nkb) {  // refill this stage once the MMAs reading it are done
        if (!mbar_wait(&bar[2 + s], ph)) ok = false;
        issue(kb + 2);
      }
    }
  }
  {
    const int last = nkb - 1;
    if (!mbar_wait(&bar[2 + (last & 1)], (last >> 1) & 1)) ok = false;
  }
  tc_fence_after();
  {
    const int wq = tid >> 5, lane = tid & 31;
    const int m = wq * 32 + lane;
    const long long bh = (long long)bi * p.H + h0 + (m >> 6);
    float* out = (kDstates ? f.dHl : f.S) + (bh * p.nc + c) * p.PN + (m & 63);
    for (int n0 = 0; n0 < p.N; n0 += 16) {
      float v[16];
      tmem_ld16(tmem_addr(tmem, wq * 32, n0), v);
#pragma unroll
      for (int j = 0; j < 16; ++j) out[(n0 + j) * 64] = v[j];
    }
  }
  if (!ok) atomicOr(&f.hdr->status, kDevTimeout);
  tc_fence_before();
  __syncthreads();
  if (tid < 32) tmem_dealloc(tmem, G.ncols);
}

}  // namespace

bool chunk_state_tc_supported(const Plan& p) {
  return p.dtype == SSD_BF16 && p.P == 64 && p.hpg % 2 == 0 && p.Q % kStageTok == 0 &&
         (p.N == 16 || p.N == 32 || p.N == 64 || p.N == 128);
}

cudaError_t launch_chunk_state_tc(const Plan& p, const Bufs& f, bool dstates, cudaStream_t s) {
  set_kernel_name(dstates ? "chunk_dstate_tc" : "chunk_state_tc");
  const StateGeom G = state_geom(p.N);
  CUtensorMap tmX, tmB;
  const uint64_t dx[4] = {(uint64_t)p.P, (uint64_t)p.H, (uint64_t)p.L, (uint64_t)p.b};
  const uint64_t sx[3] = {(uint64_t)p.P * 2, (uint64_t)p.H * p.P * 2, (uint64_t)p.L * p.H * p.P * 2};
  const uint32_t bxx[4] = {64, 1, (uint32_t)kStageTok, 1};
  const uint64_t db[4] = {(uint64_t)p.N, (uint64_t)p.G, (uint64_t)p.L, (uint64_t)p.b};
  const uint64_t sb[3] = {(uint64_t)p.N * 2, (uint64_t)p.G * p.N * 2, (uint64_t)p.L * p.G * p.N * 2};
  const uint32_t bxb[4] = {(uint32_t)(G.bw / 2), 1, (uint32_t)kStageTok, 1};
  if (!encode_tmap_bf16_4d(&tmX, dstates ? f.dy : f.x, dx, sx, bxx, 128) ||
      !encode_tmap_bf16_4d(&tmB, dstates ? f.C : f.B, db, sb, bxb, G.bw))
    return cudaErrorInvalidValue;
  const size_t smem = 1024 + 2 * (size_t)G.stage + 2 * p.Q * sizeof(float) + 64;
  auto kern = dstates ? chunk_state_tc_kernel<true> : chunk_state_tc_kernel<false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid(p.nc, p.H / 2, p.b);
  kern<<<grid, kThr, smem, s>>>(p, f, tmX, tmB);
  return cudaGetLastError();
}

}  // namespace ssd
