// k_chunk_scan_tc.cu -- chunk output on the 5th-generation tensor cores.
//
//   y_i = sum_{j<=i, seg_j=seg_i} (C_i . B_j) exp(l_i - l_j) dt_eff_j x_j     (intra-chunk)
//       + cv_i exp(l_i) H_in[c] C_i                                          (carry-in state)
//       + D_h x_i                                                            (skip)
// (page "llm-mamba-200" (gigipick.blogspot.com), section 3: the fused SSM
// block -- recurrence and output in one kernel, operands in registers and
// shared memory; the carry-in state comes from the state-passing scan).
//
// One CTA owns 128 output rows (tokens) of one chunk for all heads of one
// group.  C B^T does not depend on the head: it is formed once per CTA on
// the tensor cores (M = 128 rows, N = 128 tokens per column block J <= the
// row block, K = d_state) and stays in tensor memory.  The heads are then
// streamed: their x and carry-in-state tiles arrive by TMA into a double
// buffer while the previous head is processed; sixteen warps read C B^T back
// (one TMEM lane = one row; the four warpgroups split the columns), apply the
// causal / same-sequence mask, exp(l_i - l_j) and dt_eff_j of the head, and
// write the bf16 K-major A_hat tile; one thread issues Y1 = A_hat X and the
// carry Y2 = C H_in^T into a double-buffered accumulator pair, and the
// epilogue y = Y1 + cv e^{l} Y2 + D x of head h-1 runs while the tensor core
// works on head h.  Per-head l and dt_eff are prefetched two heads ahead
// into a ring of three shared-memory slots, the epilogue's x row one head
// ahead into registers, and 16-column blocks wholly above the diagonal for a
// warp's 32 rows are written as zeros without reading tensor memory.
#include "ssd_internal.cuh"
#include "tc_common.cuh"
#include "tma_host.h"

namespace ssd {

namespace {

using namespace tc;

constexpr int kRows = 128;  // rows (tokens i) per CTA = MMA M
constexpr int kThr = 512;   // four warpgroups: four warps per quarter of the TMEM lanes

__host__ __device__ inline uint32_t r1024(uint32_t v) { return (v + 1023u) & ~1023u; }

struct ScanGeom {
  int rows;          // tokens per TMA box = min(Q, 128)
  int nJ;            // column blocks (== number of row blocks)
  int cw, ncb;       // bytes per row of one B/C column block, column blocks along d_state
  uint32_t cblk;     // bytes of one B/C column block (kRows rows)
  uint32_t cswz;     // swizzle code of B/C tiles
  uint32_t cbytes;   // bytes of one B or C tile
  uint32_t offC, offB, offX, offH, offF, bytes;
};

__host__ __device__ inline ScanGeom scan_geom(int N, int Q) {
  ScanGeom g;
  g.rows = Q < kRows ? Q : kRows;
  g.nJ = (Q + kRows - 1) / kRows;
  g.cw = 2 * (N < 64 ? N : 64);
  g.ncb = N >= 64 ? N / 64 : 1;
  g.cblk = (uint32_t)kRows * g.cw;
  g.cswz = g.cw == 128 ? kSwz128 : (g.cw == 64 ? kSwz64 : kSwz32);
  g.cbytes = r1024(g.ncb * g.cblk);
  const uint32_t abytes = 2u * kRows * 128u;  // one 128 x 128 bf16 A_hat block
  const uint32_t bsp = g.cbytes > abytes ? g.cbytes : abytes;  // B tiles, later A_hat tiles
  g.offC = 0;
  g.offB = g.cbytes;
  g.offX = g.offB + g.nJ * bsp;                 // [2 buffers][nJ] x tiles
  g.offH = g.offX + 2u * g.nJ * kRows * 128u;   // [2 buffers] carry-in state tiles
  g.offF = g.offH + 2u * r1024((uint32_t)N * 128u);
  g.bytes = g.offF;
  return g;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

__global__ void __launch_bounds__(kThr, 1) chunk_scan_tc_kernel(Plan p, Bufs f,
                                                                const __grid_constant__ CUtensorMap tmC,
                                                                const __grid_constant__ CUtensorMap tmB,
                                                                const __grid_constant__ CUtensorMap tmX,
                                                                const __grid_constant__ CUtensorMap tmH) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const ScanGeom G = scan_geom(p.N, p.Q);
  const uint32_t abytes = 2u * kRows * 128u;
  const uint32_t bsp = G.cbytes > abytes ? G.cbytes : abytes;
  const int I = blockIdx.x % G.nJ, c = blockIdx.x / G.nJ;
  const int g = blockIdx.y, bi = blockIdx.z;
  const int tid = threadIdx.x;
  const int wg = tid >> 7;          // warpgroup: column quarter of the mask pass
  const int ri = tid & 127;         // row (TMEM lane) of this thread
  const int wlane = ((tid >> 5) & 3) * 32;
  const int t0 = c * p.Q, len = min(p.Q, p.L - t0);
  const int i0 = I * kRows;
  if (i0 >= len) return;  // row block past the ragged end (uniform per CTA)
  const int nJ = I + 1;   // column blocks J <= I
  uint8_t* sC = sm + G.offC;
  uint8_t* sB = sm + G.offB;  // B_J tiles, then A_hat_J tiles
  uint8_t* sX = sm + G.offX;
  uint8_t* sH = sm + G.offH;
  const uint32_t hbytes = r1024((uint32_t)p.N * 128u);
  float* lq = reinterpret_cast<float*>(sm + G.offF);   // [3][Q] head scalars, ring of 3 heads
  float* dq = lq + 3 * p.Q;                            // [3][Q]
  int* sq = reinterpret_cast<int*>(dq + 3 * p.Q);      // [Q]
  uint64_t* bar = reinterpret_cast<uint64_t*>(sq + p.Q);  // ld[2], mma[2], cb
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + 5);

  for (int t = tid; t < p.Q; t += kThr) sq[t] = t < len ? seg_of(p, f, bi, (long long)t0 + t) : -1;
  for (int k = 0; k < 2 && k < p.hpg; ++k) {  // scalars of the first two heads
    const long long bhk = (long long)bi * p.H + g * p.hpg + k;
    for (int t = tid; t < p.Q; t += kThr) {
      lq[k * p.Q + t] = f.lcs[bhk * p.Lp + t0 + t];
      dq[k * p.Q + t] = f.dte[bhk * p.Lp + t0 + t];
    }
  }
  if (G.rows < kRows)  // K padding rows of the x tiles must be zero
    for (int idx = tid; idx < 2 * (kRows - G.rows) * 8; idx += kThr) {
      const int buf = idx / ((kRows - G.rows) * 8), k = idx % ((kRows - G.rows) * 8);
      reinterpret_cast<uint4*>(sX + buf * G.nJ * kRows * 128 + G.rows * 128)[k] = make_uint4(0, 0, 0, 0);
    }
  if (tid == 0) {
    for (int k = 0; k < 5; ++k) mbar_init(&bar[k], 1);
    mbar_fence_init();
  }
  if (tid < 32) tmem_alloc(tmem_slot, 512);
  fence_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tm = *tmem_slot;
  const uint32_t tCB = tm;                 // nJ x 128 columns
  const uint32_t tY = tm + 256;            // [2 buffers] x (Y1 64 | Y2 64)
  bool ok = true;
  const uint32_t cbox = (uint32_t)G.rows * G.cw;
  const uint32_t xbox = (uint32_t)G.rows * 128u;
  const int hpg = p.hpg, h_first = g * hpg;

  auto issue_head = [&](int hh) {  // x tiles (J <= I) and carry-in state of head hh -> buffer hh&1
    const int buf = hh & 1, h = h_first + hh;
    mbar_expect_tx(&bar[buf], nJ * xbox + (uint32_t)p.N * 128u);
    for (int J = 0; J < nJ; ++J)
      tma_load_4d(sX + (buf * G.nJ + J) * kRows * 128, &tmX, &bar[buf], 0, h, t0 + J * kRows, bi);
    tma_load_4d(sH + buf * hbytes, &tmH, &bar[buf], 0, 0, c, bi * p.H + h);
  };
  auto mma_ck = [&](uint32_t d, const uint8_t* a, const uint8_t* b, int kdim, uint32_t idesc, bool b_mn) {
    for (int ks = 0; ks < kdim / 16; ++ks) {
      const uint32_t kb = (ks * 32) / G.cw, kin = (ks * 32) % G.cw;
      const uint64_t da = smem_desc(smem_u32(a) + kb * G.cblk + kin, 16, 8 * G.cw, G.cswz);
      const uint64_t db = b_mn ? smem_desc(smem_u32(b) + ks * 16 * 128, 16, 1024, kSwz128)
                               : smem_desc(smem_u32(b) + kb * G.cblk + kin, 16, 8 * G.cw, G.cswz);
      mma_bf16(d, da, db, idesc, ks > 0 ? 1u : 0u);
    }
  };

  // C_I and every B_J (J <= I), then CB_J = C_I B_J^T into tensor memory
  if (tid == 0) {
    mbar_expect_tx(&bar[4], (1 + nJ) * G.ncb * cbox);
    for (int q = 0; q < G.ncb; ++q) {
      tma_load_4d(sC + q * G.cblk, &tmC, &bar[4], q * 64, g, t0 + i0, bi);
      for (int J = 0; J < nJ; ++J)
        tma_load_4d(sB + J * bsp + q * G.cblk, &tmB, &bar[4], q * 64, g, t0 + J * kRows, bi);
    }
    issue_head(0);
    if (hpg > 1) issue_head(1);
  }
  if (!mbar_wait(&bar[4], 0)) ok = false;
  if (tid == 0) {
    tc_fence_after();
    for (int J = 0; J < nJ; ++J)
      mma_ck(tCB + J * 128, sC, sB + J * bsp, p.N, idesc_bf16(128, 128, 0, 0), false);
    mma_commit(&bar[4]);
  }
  if (!mbar_wait(&bar[4], 1)) ok = false;
  tc_fence_after();
  // from here on the B tiles' space holds the A_hat tiles

  const int i = i0 + ri;
  const bool row_ok = i < len;
  const int si = row_ok ? sq[i] : -2;
  const int s_in = seg_in_of(p, f, bi, c);
  __nv_bfloat16* y = static_cast<__nv_bfloat16*>(f.y);
  const __nv_bfloat16* xg = static_cast<const __nv_bfloat16*>(f.x);

  // x row of head hh for the skip term (this thread's row, its 32 columns),
  // fetched one iteration ahead of its use
  auto fetch_x = [&](int hh, uint4 (&xv)[2]) {
    const long long xrow = (((long long)bi * p.L + t0 + i) * p.H + h_first + hh) * 64 + wg * 16;
    const uint4* xr = reinterpret_cast<const uint4*>(xg + xrow);
    xv[0] = row_ok ? xr[0] : make_uint4(0, 0, 0, 0);
    xv[1] = row_ok ? xr[1] : make_uint4(0, 0, 0, 0);
  };
  // y rows of head hh from accumulator buffer hh&1; li is the row's l of head
  // hh, kept in a register from the mask pass (its ring slot is refilled in
  // the same iteration as this epilogue runs)
  auto epilogue = [&](int hh, const uint4 (&xv)[2], float li) {
    const int buf = hh & 1, h = h_first + hh;
    const float carry = (row_ok && si == s_in) ? __expf(li) : 0.0f;
    const float Dh = f.D[h];
    const long long yrow = (((long long)bi * p.L + t0 + i) * p.H + h) * 64;
    {
      const int q = wg;  // the four warpgroups split the 64 output columns
      float a[16], b[16];
      tmem_ld16x2(tmem_addr(tY + buf * 128, wlane, q * 16), tmem_addr(tY + buf * 128 + 64, wlane, q * 16), a, b);
      if (row_ok) {
        const uint4 x0 = xv[0], x1 = xv[1];
        const uint32_t xs[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
        uint32_t o[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float2 xf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&xs[e]));
          o[e] = pack_bf16x2(a[2 * e] + carry * b[2 * e] + Dh * xf.x,
                             a[2 * e + 1] + carry * b[2 * e + 1] + Dh * xf.y);
        }
        uint4* dst = reinterpret_cast<uint4*>(y + yrow + q * 16);
        dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
        dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
      }
    }
  };

  uint4 xprev[2] = {};
  float li_prev = 0.0f;  // l of the head whose epilogue is pending
  for (int hh = 0; hh < hpg; ++hh) {
    const int buf = hh & 1;
    // prefetch, for later in this iteration: the x row of head hh-1 (epilogue)
    // and the scalars of head hh+2 (ring slot (hh+2)%3, last read by head hh-1)
    uint4 xcur[2];
    if (hh > 0) fetch_x(hh - 1, xcur);
    const int pre = hh + 2;
    float pl = 0.0f, pd = 0.0f;
    const int tq = tid;  // Q <= 256 < kThr: one scalar pair per thread
    if (pre < hpg && tq < p.Q) {
      const long long bhp = (long long)bi * p.H + h_first + pre;
      pl = f.lcs[bhp * p.Lp + t0 + tq];
      pd = f.dte[bhp * p.Lp + t0 + tq];
    }
    if (hh > 0) {  // MMAs of head hh-1 done: A_hat and the other buffers are free
      if (!mbar_wait(&bar[2 + ((hh - 1) & 1)], ((hh - 1) >> 1) & 1)) ok = false;
      tc_fence_after();
      if (tid == 0 && hh + 1 < hpg) issue_head(hh + 1);
    }
    __syncthreads();
    {  // mask pass: row ri, column half wg of every block J
      const float* lb = lq + (hh % 3) * p.Q;
      const float* db = dq + (hh % 3) * p.Q;
      const float li = row_ok ? lb[i] : 0.0f;
      const int warp_last_row = i0 + wlane + 31;  // last row of this warp
      for (int J = 0; J < nJ; ++J) {
        uint8_t* aJ = sB + J * bsp;
        for (int q = wg * 2; q < wg * 2 + 2; ++q) {
          uint32_t pk[8] = {0, 0, 0, 0, 0, 0, 0, 0};
          if (J * kRows + q * 16 <= warp_last_row && J * kRows + q * 16 < len) {  // else all masked
            float v[16];
            tmem_ld16(tmem_addr(tCB + J * 128, wlane, q * 16), v);
#pragma unroll
            for (int e = 0; e < 16; e += 2) {
              float a2[2];
#pragma unroll
              for (int u = 0; u < 2; ++u) {
                const int j = J * kRows + q * 16 + e + u;
                a2[u] = (row_ok && j <= i && sq[j] == si) ? v[e + u] * __expf(li - lb[j]) * db[j] : 0.0f;
              }
              pk[e / 2] = pack_bf16x2(a2[0], a2[1]);
            }
          }
          uint8_t* blk = aJ + (q / 4) * (kRows * 128);
          const uint32_t e0 = (q % 4) * 16;
          *reinterpret_cast<uint4*>(blk + swz128_off(ri, e0)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
          *reinterpret_cast<uint4*>(blk + swz128_off(ri, e0 + 8)) = make_uint4(pk[4], pk[5], pk[6], pk[7]);
        }
      }
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    if (tid == 0) {
      if (!mbar_wait(&bar[buf], (hh >> 1) & 1)) ok = false;  // x and state tiles of head hh
      tc_fence_after();
      const uint32_t d1 = tY + buf * 128, d2 = d1 + 64;
      const uint32_t id64 = idesc_bf16(128, 64, 0, 1);
      const uint8_t* xb = sX + buf * G.nJ * kRows * 128;
      for (int J = 0; J < nJ; ++J)
        for (int ks = 0; ks < kRows / 16; ++ks) {  // Y1 += A_hat_J X_J
          const uint64_t da =
              smem_desc(smem_u32(sB + J * bsp) + (ks / 4) * (kRows * 128) + (ks % 4) * 32, 16, 1024, kSwz128);
          const uint64_t dbx = smem_desc(smem_u32(xb + J * kRows * 128) + ks * 16 * 128, 16, 1024, kSwz128);
          mma_bf16(d1, da, dbx, id64, (J > 0 || ks > 0) ? 1u : 0u);
        }
      mma_ck(d2, sC, sH + buf * hbytes, p.N, id64, true);  // Y2 = C_I H^T
      mma_commit(&bar[2 + buf]);
    }
    if (hh > 0) epilogue(hh - 1, xcur, li_prev);
    li_prev = row_ok ? lq[(hh % 3) * p.Q + i] : 0.0f;
    if (pre < hpg && tq < p.Q) {
      lq[(pre % 3) * p.Q + tq] = pl;
      dq[(pre % 3) * p.Q + tq] = pd;
    }
  }
  {
    const int last = hpg - 1;
    fetch_x(last, xprev);
    if (!mbar_wait(&bar[2 + (last & 1)], (last >> 1) & 1)) ok = false;
    tc_fence_after();
    epilogue(last, xprev, li_prev);
  }
  if (!ok) atomicOr(&f.hdr->status, kDevTimeout);
  tc_fence_before();
  __syncthreads();
  if (tid < 32) tmem_dealloc(tm, 512);
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
  const size_t smem = 1024 + G.bytes + 7 * p.Q * 4 + 64;
  cudaError_t e = cudaFuncSetAttribute(chunk_scan_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid(p.nc * G.nJ, p.G, p.b);
  chunk_scan_tc_kernel<<<grid, kThr, smem, s>>>(p, f, tmC, tmB, tmX, tmH);
  return cudaGetLastError();
}

}  // namespace ssd
