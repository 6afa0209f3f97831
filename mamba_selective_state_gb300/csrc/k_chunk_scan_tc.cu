// k_chunk_scan_tc.cu -- chunk output on the 5th-generation tensor cores.
//
//   y_i = sum_{j<=i, seg_j=seg_i} (C_i . B_j) exp(l_i - l_j) dt_eff_j x_j     (intra-chunk)
//       + cv_i exp(l_i) H_in[c] C_i                                          (carry-in state)
//       + D_h x_i                                                            (skip)
// (page "llm-mamba-200" (gigipick.blogspot.com), section 3: the fused SSM
// block -- recurrence and output in one kernel, operands in registers and
// shared memory; the carry-in state comes from the state-passing scan).
//
// One CTA owns 128 output rows (tokens) of one chunk of one head.  For every
// 128-token column block J <= the row block:
//   1. CB = C_I B_J^T on the tensor cores (M = 128 rows, N = 128 tokens,
//      K = d_state) into tensor memory;
//   2. the four warps read CB back (one TMEM lane = one row per thread),
//      apply the causal / same-sequence mask, exp(l_i - l_j) and dt_eff_j, and
//      write the bf16 result as the K-major A operand in shared memory;
//   3. Y1 += A_hat X_J (N = headdim 64, K = 128 tokens).
// The carry term Y2 = C_I H_in^T (K = d_state) goes to a second accumulator;
// the epilogue forms y = Y1 + cv_i e^{l_i} Y2 + D_h x_i and stores bf16.
// Operands arrive by TMA with 128-byte swizzle (narrower for d_state < 64).
#include "ssd_internal.cuh"
#include "tc_common.cuh"
#include "tma_host.h"

namespace ssd {

namespace {

using namespace tc;

constexpr int kRows = 128;  // rows (tokens i) per CTA = MMA M
constexpr int kThr = 128;

__host__ __device__ inline uint32_t r1024(uint32_t v) { return (v + 1023u) & ~1023u; }

struct ScanGeom {
  int rows;          // tokens per TMA box = min(Q, 128)
  int cw;            // bytes per row of one B/C column block (2 * min(N, 64))
  int ncb;           // column blocks along d_state
  uint32_t cblk;     // bytes of one B/C column block (kRows rows)
  uint32_t cswz;     // swizzle code of B/C tiles
  uint32_t offC, offB, offA, offX, offH, offF;  // smem offsets (A_hat may alias B)
  uint32_t bytes;
};

__host__ __device__ inline ScanGeom scan_geom(int N, int Q) {
  ScanGeom g;
  g.rows = Q < kRows ? Q : kRows;
  g.cw = 2 * (N < 64 ? N : 64);
  g.ncb = N >= 64 ? N / 64 : 1;
  g.cblk = (uint32_t)kRows * g.cw;
  g.cswz = g.cw == 128 ? kSwz128 : (g.cw == 64 ? kSwz64 : kSwz32);
  const uint32_t cbytes = r1024(g.ncb * g.cblk);
  const uint32_t abytes = 2u * kRows * 128u;  // 128 x 128 bf16, two 64-column blocks
  g.offC = 0;
  g.offB = cbytes;
  g.offA = cbytes >= abytes ? g.offB : g.offB + cbytes;  // A_hat reuses B when it fits
  const uint32_t endBA = (g.offA == g.offB) ? g.offB + cbytes : g.offA + abytes;
  g.offX = endBA;
  g.offH = g.offX + kRows * 128u;
  g.offF = g.offH + r1024((uint32_t)N * 128u);
  g.bytes = g.offF;
  return g;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

__global__ void __launch_bounds__(kThr) chunk_scan_tc_kernel(Plan p, Bufs f,
                                                             const __grid_constant__ CUtensorMap tmC,
                                                             const __grid_constant__ CUtensorMap tmB,
                                                             const __grid_constant__ CUtensorMap tmX,
                                                             const __grid_constant__ CUtensorMap tmH) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const ScanGeom G = scan_geom(p.N, p.Q);
  const int nI = (p.Q + kRows - 1) / kRows;
  const int c = blockIdx.x / nI, I = blockIdx.x - c * nI;
  const int h = blockIdx.y, bi = blockIdx.z;
  const int g = h / p.hpg;
  const int tid = threadIdx.x;
  const int t0 = c * p.Q, len = min(p.Q, p.L - t0);
  const long long bh = (long long)bi * p.H + h;
  uint8_t* sC = sm + G.offC;
  uint8_t* sB = sm + G.offB;
  uint8_t* sA = sm + G.offA;
  uint8_t* sX = sm + G.offX;
  uint8_t* sH = sm + G.offH;
  float* lq = reinterpret_cast<float*>(sm + G.offF);   // [Q]
  float* dq = lq + p.Q;                                // [Q]
  int* sq = reinterpret_cast<int*>(dq + p.Q);          // [Q]
  uint64_t* bar = reinterpret_cast<uint64_t*>(sq + p.Q);  // load, mma
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + 2);
  const int i0 = I * kRows;
  if (i0 >= len) return;  // block past the ragged end (uniform per CTA)

  for (int i = tid; i < p.Q; i += kThr) {
    lq[i] = f.lcs[bh * p.Lp + t0 + i];
    dq[i] = f.dte[bh * p.Lp + t0 + i];
    sq[i] = i < len ? seg_of(p, f, bi, (long long)t0 + i) : -1;
  }
  // rows of the x tile beyond the chunk are the K padding of the intra MMA:
  // make them zero (the TMA box covers only min(Q, 128) rows)
  if (G.rows < kRows)
    for (int idx = tid; idx < (kRows - G.rows) * 8; idx += kThr)
      reinterpret_cast<uint4*>(sX + G.rows * 128)[idx] = make_uint4(0, 0, 0, 0);
  if (tid == 0) {
    mbar_init(&bar[0], 1);
    mbar_init(&bar[1], 1);
    mbar_fence_init();
  }
  if (tid < 32) tmem_alloc(tmem_slot, 256);
  fence_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tCB = tmem, tY1 = tmem + 128, tY2 = tmem + 192;
  bool ok = true;
  uint32_t ld_phase = 0, mma_phase = 0;
  const uint32_t cbox = (uint32_t)G.rows * G.cw;

  auto load_bx = [&](int J, bool withCH) {
    uint32_t bytes = G.ncb * cbox + (uint32_t)G.rows * 128u;
    if (withCH) bytes += G.ncb * cbox + (uint32_t)p.N * 128u;
    mbar_expect_tx(&bar[0], bytes);
    for (int q = 0; q < G.ncb; ++q) tma_load_4d(sB + q * G.cblk, &tmB, &bar[0], q * 64, g, t0 + J * kRows, bi);
    tma_load_4d(sX, &tmX, &bar[0], 0, h, t0 + J * kRows, bi);
    if (withCH) {
      for (int q = 0; q < G.ncb; ++q) tma_load_4d(sC + q * G.cblk, &tmC, &bar[0], q * 64, g, t0 + i0, bi);
      tma_load_4d(sH, &tmH, &bar[0], 0, 0, c, (int)bh);
    }
  };
  auto mma_ck = [&](uint32_t d, uint8_t* a, uint8_t* b, int kdim, uint32_t idesc, bool b_mn,
                    bool acc0) {
    // A: K-major C-like tile (d_state columns); B: K-major (b_mn=false) or the
    // MN-major H tile (b_mn=true)
    for (int ks = 0; ks < kdim / 16; ++ks) {
      const uint32_t kb = (ks * 32) / G.cw, kin = (ks * 32) % G.cw;
      const uint64_t da = smem_desc(smem_u32(a) + kb * G.cblk + kin, 16, 8 * G.cw, G.cswz);
      const uint64_t db = b_mn ? smem_desc(smem_u32(b) + ks * 16 * 128, 16, 1024, kSwz128)
                               : smem_desc(smem_u32(b) + kb * G.cblk + kin, 16, 8 * G.cw, G.cswz);
      mma_bf16(d, da, db, idesc, (acc0 || ks > 0) ? 1u : 0u);
    }
  };

  if (tid == 0) load_bx(0, true);
  const int ri = tid;                 // this thread's row (TMEM lane) within the block
  const int i = i0 + ri;              // chunk-local token
  const bool row_ok = i < len;
  const float li = row_ok ? lq[i] : 0.0f;
  const int si = row_ok ? sq[i] : -2;
  const int s_in = seg_in_of(p, f, bi, c);

  for (int J = 0; J <= I; ++J) {
    if (J > 0 && tid == 0) load_bx(J, false);
    if (!mbar_wait(&bar[0], ld_phase)) ok = false;
    ld_phase ^= 1;
    if (tid == 0) {
      tc_fence_after();
      if (J == 0)  // carry: Y2 = C_I H^T  (M 128, N 64, K d_state)
        mma_ck(tY2, sC, sH, p.N, idesc_bf16(128, 64, 0, 1), true, false);
      mma_ck(tCB, sC, sB, p.N, idesc_bf16(128, 128, 0, 0), false, false);  // CB = C_I B_J^T
      mma_commit(&bar[1]);
    }
    if (!mbar_wait(&bar[1], mma_phase)) ok = false;
    mma_phase ^= 1;
    tc_fence_after();
    // mask + decay + dt, bf16, into the K-major A_hat tile (row ri)
    for (int q = 0; q < kRows / 16; ++q) {
      float v[16];
      tmem_ld16(tmem_addr(tCB, (tid >> 5) * 32, q * 16), v);
      uint32_t pk[8];
#pragma unroll
      for (int e = 0; e < 16; e += 2) {
        float a2[2];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int j = J * kRows + q * 16 + e + u;
          float val = 0.0f;
          if (row_ok && j <= i && sq[j] == si) val = v[e + u] * __expf(li - lq[j]) * dq[j];
          a2[u] = val;
        }
        pk[e / 2] = pack_bf16x2(a2[0], a2[1]);
      }
      const int col = q * 16;  // first column (token j within block J)
      uint8_t* blk = sA + (col / 64) * (kRows * 128);
      const uint32_t e0 = col % 64;
      *reinterpret_cast<uint4*>(blk + swz128_off(ri, e0)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
      *reinterpret_cast<uint4*>(blk + swz128_off(ri, e0 + 8)) = make_uint4(pk[4], pk[5], pk[6], pk[7]);
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    if (tid == 0) {
      tc_fence_after();
      const uint32_t idesc = idesc_bf16(128, 64, 0, 1);
      for (int ks = 0; ks < kRows / 16; ++ks) {  // Y1 += A_hat X_J (K = 128 tokens)
        const uint64_t da = smem_desc(smem_u32(sA) + (ks / 4) * (kRows * 128) + (ks % 4) * 32, 16, 1024, kSwz128);
        const uint64_t db = smem_desc(smem_u32(sX) + ks * 16 * 128, 16, 1024, kSwz128);
        mma_bf16(tY1, da, db, idesc, (J > 0 || ks > 0) ? 1u : 0u);
      }
      mma_commit(&bar[1]);
    }
    if (!mbar_wait(&bar[1], mma_phase)) ok = false;  // A_hat, B and X are free again
    mma_phase ^= 1;
    tc_fence_after();
  }
  // epilogue: y = Y1 + cv e^{l} Y2 + D x  (x row ri of the last X tile = block I)
  {
    const float carry = (row_ok && si == s_in) ? __expf(li) : 0.0f;
    const float Dh = f.D[h];
    __nv_bfloat16* y = static_cast<__nv_bfloat16*>(f.y);
    const long long yrow = (((long long)bi * p.L + t0 + i) * p.H + h) * 64;
    for (int q = 0; q < 4; ++q) {
      float a[16], b[16];
      tmem_ld16(tmem_addr(tY1, (tid >> 5) * 32, q * 16), a);
      tmem_ld16(tmem_addr(tY2, (tid >> 5) * 32, q * 16), b);
      const uint4 x0 = *reinterpret_cast<const uint4*>(sX + swz128_off(ri, q * 16));
      const uint4 x1 = *reinterpret_cast<const uint4*>(sX + swz128_off(ri, q * 16 + 8));
      const uint32_t xs[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
      uint32_t o[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float2 xf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&xs[e]));
        o[e] = pack_bf16x2(a[2 * e] + carry * b[2 * e] + Dh * xf.x,
                           a[2 * e + 1] + carry * b[2 * e + 1] + Dh * xf.y);
      }
      if (row_ok) {
        uint4* dst = reinterpret_cast<uint4*>(y + yrow + q * 16);
        dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
        dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
      }
    }
  }
  if (!ok) atomicOr(&f.hdr->status, kDevTimeout);
  tc_fence_before();
  __syncthreads();
  if (tid < 32) tmem_dealloc(tmem, 256);
}

}  // namespace

bool chunk_scan_tc_supported(const Plan& p) {
  return p.dtype == SSD_BF16 && p.P == 64 && (p.Q == 64 || p.Q == 128 || p.Q == 256) &&
         (p.N == 16 || p.N == 32 || p.N == 64 || p.N == 128);
}

cudaError_t launch_chunk_scan_tc(const Plan& p, const Bufs& f, cudaStream_t s) {
  set_kernel_name("chunk_scan_tc");
  const ScanGeom G = scan_geom(p.N, p.Q);
  CUtensorMap tmC, tmB, tmX, tmH;
  const uint32_t rows = (uint32_t)G.rows;
  const uint64_t dbc[4] = {(uint64_t)p.N, (uint64_t)p.G, (uint64_t)p.L, (uint64_t)p.b};
  const uint64_t sbc[3] = {(uint64_t)p.N * 2, (uint64_t)p.G * p.N * 2, (uint64_t)p.L * p.G * p.N * 2};
  const uint32_t bbc[4] = {(uint32_t)(G.cw / 2), 1, rows, 1};
  const uint64_t dxx[4] = {64, (uint64_t)p.H, (uint64_t)p.L, (uint64_t)p.b};
  const uint64_t sxx[3] = {128, (uint64_t)p.H * 128, (uint64_t)p.L * p.H * 128};
  const uint32_t bxx[4] = {64, 1, rows, 1};
  // carry-in states (b*H, nc, N, 64) bf16
  const uint64_t dh[4] = {64, (uint64_t)p.N, (uint64_t)p.nc, (uint64_t)p.b * p.H};
  const uint64_t sh[3] = {128, (uint64_t)p.N * 128, (uint64_t)p.nc * p.N * 128};
  const uint32_t bh[4] = {64, (uint32_t)p.N, 1, 1};
  if (!encode_tmap_bf16_4d(&tmC, f.C, dbc, sbc, bbc, G.cw) ||
      !encode_tmap_bf16_4d(&tmB, f.B, dbc, sbc, bbc, G.cw) ||
      !encode_tmap_bf16_4d(&tmX, f.x, dxx, sxx, bxx, 128) ||
      !encode_tmap_bf16_4d(&tmH, f.Hin, dh, sh, bh, 128))
    return cudaErrorInvalidValue;
  const size_t smem = 1024 + G.bytes + 3 * p.Q * 4 + 64;
  cudaError_t e = cudaFuncSetAttribute(chunk_scan_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  const int nI = (p.Q + kRows - 1) / kRows;
  dim3 grid(p.nc * nI, p.H, p.b);
  chunk_scan_tc_kernel<<<grid, kThr, smem, s>>>(p, f, tmC, tmB, tmX, tmH);
  return cudaGetLastError();
}

}  // namespace ssd
