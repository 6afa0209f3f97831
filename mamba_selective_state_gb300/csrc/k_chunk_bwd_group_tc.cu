// k_chunk_bwd_group_tc.cu -- per-head token gradients of one chunk for all
// heads of one group, on the 5th-generation tensor cores (chunk <= 128).
//
// Notation (chunk c, head h, chunk-local tokens i, j):
//   E_ij = exp(l_i - l_j) [j <= i, seg_i = seg_j],  M_ij = (C_i.B_j) E_ij dt_j,
//   dM_ij = dy_i . x_j,  R_ij = dM_ij M_ij,  u_j = sv_j exp(l_last - l_j) dt_j.
// Writes, per head:
//   dx_j      = sum_i M_ij dy_i + u_j dS B_j + D_h dy_j
//   ddt_eff_j = sum_i dM_ij (C_i.B_j) E_ij + sv_j exp(l_last - l_j) (x_j . dS B_j)
//   dl_t      = sum_j R_tj - sum_i R_it + [cv_t] e^{l_t} dy_t . (H C_t) - u_t (x_t . dS B_t)
// and the per-chunk partials sum_j u_j (x_j . dS B_j) and sum dy . x.
//
// One CTA (512 threads: 16 warps, four per quarter of the tensor-memory
// lanes) per (chunk, group, batch row).  C B^T does not depend on the head: it
// is formed once and stays in tensor memory.  For each head of the group
// (x, dy double-buffered by TMA; dS, H single-buffered):
//   1. tensor cores: dM = dy x^T (M = i), dXs = B dS^T, Yc = C H^T -- issued
//      while the previous head's epilogue runs (dXs is double-buffered);
//   2. the warps read C B^T and dM back (thread = row i; the four warpgroups
//      split the columns), form E, M, R and dM (C.B) E; row sums stay in the
//      thread; column sums are taken by a fixed warp-shuffle transpose-reduce
//      and a fixed-order fold over the lane quarters (bitwise reproducible);
//      M is written row by row as a bf16 tile that the tensor core reads as
//      the MN-major A operand of M^T; 16-column blocks that lie wholly above
//      the diagonal for a warp's 32 rows are skipped;
//   3. tensor cores: dX = M^T dy (M = j);
//   4. epilogue (thread = token j): dx, ddt_eff, dl to global memory; the
//      per-chunk sums are warp butterflies folded in a fixed order.
// (page "B200 Helion Mamba-2" (aitrends.kr/articles/109906), section "Helion
// based B200 kernel redesign": TMA, TMEM and warp specialisation on
// Blackwell; page "flashinfer PR 6997 Cake RMSNorm" (blog.secrett2633.cloud),
// section "Fixed-order Tree Fold Reduction": deterministic reductions.)
#include "ssd_internal.cuh"
#include "tc_common.cuh"
#include "tma_host.h"

namespace ssd {

namespace {

using namespace tc;

constexpr int kRows = 128;
constexpr int kThr = 512;  // 16 warps: four read each quarter of the tensor-memory lanes
constexpr float kLog2e = 1.4426950408889634f;
constexpr unsigned kFull = 0xffffffffu;
constexpr uint32_t kTok = kRows * 128u;  // one (128 tokens x 64) bf16 tile

__host__ __device__ inline uint32_t r1024(uint32_t v) { return (v + 1023u) & ~1023u; }

struct GTiles {
  int rows, cw, ncb;
  uint32_t cblk, cswz, cbytes, sbytes;
  uint32_t offB, offC, offA, offX, offY, offS, offH, offF;
};

__host__ __device__ inline GTiles gtiles(int N, int Q) {
  GTiles t;
  t.rows = Q < kRows ? Q : kRows;
  t.cw = 2 * (N < 64 ? N : 64);
  t.ncb = N >= 64 ? N / 64 : 1;
  t.cblk = (uint32_t)kRows * t.cw;
  t.cswz = t.cw == 128 ? kSwz128 : (t.cw == 64 ? kSwz64 : kSwz32);
  t.cbytes = r1024(t.ncb * t.cblk);
  t.sbytes = r1024((uint32_t)N * 128u);
  t.offB = 0;
  t.offC = t.cbytes;
  t.offA = 2 * t.cbytes;              // M tile, 128 x 128 bf16 (two 64-column blocks)
  t.offX = t.offA + 2 * kTok;         // [2] x tiles
  t.offY = t.offX + 2 * kTok;         // [2] dy tiles
  t.offS = t.offY + 2 * kTok;         // dS tile
  t.offH = t.offS + t.sbytes;         // H tile
  t.offF = t.offH + t.sbytes;
  return t;
}

__device__ __forceinline__ uint32_t pack2(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}
__device__ __forceinline__ float2 unpack2(uint32_t v) {
  return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&v));
}

// Column sums of a 32-row x 16-column block held one row per lane: after the
// call, lane l holds the sum over the warp's 32 rows of column
// 8*b4 + 4*b3 + 2*b2 + b1 (b_k = bit k of l).  Fixed butterfly order.
__device__ __forceinline__ float colsum16(float (&v)[16], int lane) {
  float a8[8];
  const bool hi16 = lane & 16;
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const float send = hi16 ? v[k] : v[8 + k];
    const float keep = hi16 ? v[8 + k] : v[k];
    a8[k] = keep + __shfl_xor_sync(kFull, send, 16);
  }
  float a4[4];
  const bool hi8 = lane & 8;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float send = hi8 ? a8[k] : a8[4 + k];
    const float keep = hi8 ? a8[4 + k] : a8[k];
    a4[k] = keep + __shfl_xor_sync(kFull, send, 8);
  }
  float a2[2];
  const bool hi4 = lane & 4;
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const float send = hi4 ? a4[k] : a4[2 + k];
    const float keep = hi4 ? a4[2 + k] : a4[k];
    a2[k] = keep + __shfl_xor_sync(kFull, send, 4);
  }
  const bool hi2 = lane & 2;
  const float send = hi2 ? a2[0] : a2[1];
  const float keep = hi2 ? a2[1] : a2[0];
  float a1 = keep + __shfl_xor_sync(kFull, send, 2);
  a1 += __shfl_xor_sync(kFull, a1, 1);
  return a1;
}

__device__ __forceinline__ bool wait_mma(uint64_t* bar, uint32_t& ph) {
  const bool r = mbar_wait(bar, ph);
  ph ^= 1;
  tc_fence_after();
  return r;
}

// Butterfly sum over the 32 lanes, in a fixed order.
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
  return v;
}

// Rows beyond a short chunk (chunk < 128) of the x, dy, B and C tiles are
// never written by the tensor copies: zero them once, so that they add
// exact zeros wherever a contraction runs over tokens.
__device__ __forceinline__ void zero_padding(const GTiles& T, uint8_t* sXb, uint8_t* sYb, uint8_t* sB,
                                             uint8_t* sC, int tid) {
  if (T.rows >= kRows) return;
  for (int idx = tid; idx < 4 * (kRows - T.rows) * 8; idx += kThr) {
    const int which = idx / ((kRows - T.rows) * 8), k = idx % ((kRows - T.rows) * 8);
    uint8_t* base = (which < 2 ? sXb : sYb) + (which & 1) * kTok + T.rows * 128;
    reinterpret_cast<uint4*>(base)[k] = make_uint4(0, 0, 0, 0);
  }
  const int per = (kRows - T.rows) * T.cw / 16;
  for (int idx = tid; idx < 2 * T.ncb * per; idx += kThr) {
    const int blk = idx / per, k = idx % per;
    uint8_t* base = (blk < T.ncb ? sB : sC) + (blk % T.ncb) * T.cblk + T.rows * T.cw;
    reinterpret_cast<uint4*>(base)[k] = make_uint4(0, 0, 0, 0);
  }
}

// Shared-memory words after the tiles: l*log2(e) and dt of two heads, the
// segment ids, the partial-sum arrays of the token kernel, then barriers.
__host__ __device__ inline size_t group_smem_bytes(const GTiles& T, int Q) {
  return 1024 + T.offF + (size_t)(5 * Q + 24 * kRows + 8) * 4 + 8 * 8 + 16;
}

__global__ void __launch_bounds__(kThr, 1) chunk_bwd_group_tc_kernel(Plan p, Bufs f,
                                                                    const __grid_constant__ CUtensorMap tmX,
                                                                    const __grid_constant__ CUtensorMap tmY,
                                                                    const __grid_constant__ CUtensorMap tmB,
                                                                    const __grid_constant__ CUtensorMap tmC,
                                                                    const __grid_constant__ CUtensorMap tmS,
                                                                    const __grid_constant__ CUtensorMap tmH) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const GTiles T = gtiles(p.N, p.Q);
  uint8_t* sB = sm + T.offB;
  uint8_t* sC = sm + T.offC;
  uint8_t* sA = sm + T.offA;
  uint8_t* sXb = sm + T.offX;
  uint8_t* sYb = sm + T.offY;
  uint8_t* sS = sm + T.offS;
  uint8_t* sH = sm + T.offH;
  float* l2q = reinterpret_cast<float*>(sm + T.offF);  // [2 slots][Q] l * log2(e) of a head
  float* dtq = l2q + 2 * p.Q;                         // [2 slots][Q] dt of a head
  int* sq = reinterpret_cast<int*>(dtq + 2 * p.Q);    // [Q] segment ids
  float* colR = reinterpret_cast<float*>(sq + p.Q);   // [4 lane quarters][128] column sums of R
  float* colQ = colR + 4 * kRows;                     // [4][128] column sums of dM (C.B) E
  float* rowR = colQ + 4 * kRows;                     // [4 warpgroups][128] row sums of R
  float* carP = rowR + 4 * kRows;                     // [4][128] carry term of dl, by headdim quarter
  float* duP = carP + 4 * kRows;                      // [4][128] x . dS B, by headdim quarter
  float* dyxP = duP + 4 * kRows;                      // [4][128] dy . x, by headdim quarter
  float* red = dyxP + 4 * kRows;                      // [8] per-warp sums
  uint64_t* bar = reinterpret_cast<uint64_t*>(red + 8);  // ld_bc, ld_xy[2], ld_sh, batch1, dX
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + 6);

  const int c = blockIdx.x, g = blockIdx.y, bi = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31;
  const int wg = tid >> 7, r = tid & 127, wq = (tid >> 5) & 3;
  const int wlane = wq * 32;
  const int t0 = c * p.Q, len = min(p.Q, p.L - t0);
  const int hpg = p.hpg, h_first = g * hpg;
  const long long bh0 = (long long)bi * p.H + h_first;

  for (int t = tid; t < p.Q; t += kThr) sq[t] = t < len ? seg_of(p, f, bi, (long long)t0 + t) : -1;
  if (tid < p.Q) {  // scalars of the group's first head into slot 0
    l2q[tid] = f.lcs[bh0 * p.Lp + t0 + tid] * kLog2e;
    dtq[tid] = f.dte[bh0 * p.Lp + t0 + tid];
  }
  zero_padding(T, sXb, sYb, sB, sC, tid);
  if (tid == 0) {
    for (int k = 0; k < 6; ++k) mbar_init(&bar[k], 1);
    mbar_fence_init();
  }
  if (tid < 32) tmem_alloc(tmem_slot, 512);
  fence_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tm = *tmem_slot;
  // C B^T | dM | dX | dXs (two buffers) | Yc
  const uint32_t tCB = tm, tDM = tm + 128, tDX = tm + 256, tDXS = tm + 320, tYC = tm + 448;
  const int s_in = seg_in_of(p, f, bi, c);
  const int s_last = sq[len - 1];
  const bool one_seg = sq[0] == s_last;  // seq_idx is nondecreasing: no reset inside the chunk
  bool ok = true;
  uint32_t ph_m1 = 0, ph_m2 = 0;
  const uint32_t tok_bytes = (uint32_t)T.rows * 128u;
  const uint32_t c_bytes = (uint32_t)T.ncb * T.rows * T.cw;
  const uint32_t s_bytes = (uint32_t)p.N * 128u;
  const uint32_t id128 = idesc_bf16(128, 128, 0, 0), id64 = idesc_bf16(128, 64, 0, 1);
  const uint32_t id64t = idesc_bf16(128, 64, 1, 1);

  auto issue_xy = [&](int hh) {
    const int buf = hh & 1, h = h_first + hh;
    mbar_expect_tx(&bar[1 + buf], 2 * tok_bytes);
    tma_load_4d(sXb + buf * kTok, &tmX, &bar[1 + buf], 0, h, t0, bi);
    tma_load_4d(sYb + buf * kTok, &tmY, &bar[1 + buf], 0, h, t0, bi);
  };
  auto issue_sh = [&](int hh) {
    const int h = h_first + hh;
    mbar_expect_tx(&bar[3], 2 * s_bytes);
    tma_load_4d(sS, &tmS, &bar[3], 0, 0, c, bi * p.H + h);
    tma_load_4d(sH, &tmH, &bar[3], 0, 0, c, bi * p.H + h);
  };
  auto kdesc_c = [&](const uint8_t* t, int ks) {  // K-major B/C tile, K = d_state
    const uint32_t kb = (ks * 32) / T.cw, kin = (ks * 32) % T.cw;
    return smem_desc(smem_u32(t) + kb * T.cblk + kin, 16, 8 * T.cw, T.cswz);
  };
  auto kdesc_tok = [&](const uint8_t* t, int ks) {  // K-major 128 x 64 token tile, K = 64
    return smem_desc(smem_u32(t) + ks * 32, 16, 1024, kSwz128);
  };
  auto mndesc_rows = [&](const uint8_t* t, int ks) {  // MN-major (64 wide), K along rows
    return smem_desc(smem_u32(t) + ks * 16 * 128, 16, 1024, kSwz128);
  };
  // batch 1 of head hh: dM = dy x^T, dXs = B dS^T (buffer hh&1), Yc = C H^T
  auto batch1 = [&](int hh) {
    const int buf = hh & 1;
    const uint8_t* sX = sXb + buf * kTok;
    const uint8_t* sY = sYb + buf * kTok;
    for (int ks = 0; ks < 4; ++ks) mma_bf16(tDM, kdesc_tok(sY, ks), kdesc_tok(sX, ks), id128, ks > 0);
    for (int ks = 0; ks < p.N / 16; ++ks) {
      mma_bf16(tDXS + buf * 64, kdesc_c(sB, ks), mndesc_rows(sS, ks), id64, ks > 0);
      mma_bf16(tYC, kdesc_c(sC, ks), mndesc_rows(sH, ks), id64, ks > 0);
    }
    mma_commit(&bar[4]);
  };

  if (tid == 0) {
    mbar_expect_tx(&bar[0], 2 * c_bytes);
    for (int q = 0; q < T.ncb; ++q) {
      tma_load_4d(sB + q * T.cblk, &tmB, &bar[0], q * 64, g, t0, bi);
      tma_load_4d(sC + q * T.cblk, &tmC, &bar[0], q * 64, g, t0, bi);
    }
    issue_xy(0);
    if (hpg > 1) issue_xy(1);
    issue_sh(0);
    if (!mbar_wait(&bar[0], 0)) ok = false;
    tc_fence_after();
    for (int ks = 0; ks < p.N / 16; ++ks)  // C B^T (M = i, N = j, K = d_state), once per group
      mma_bf16(tCB, kdesc_c(sC, ks), kdesc_c(sB, ks), id128, ks > 0);
    if (!mbar_wait(&bar[1], 0)) ok = false;
    if (!mbar_wait(&bar[3], 0)) ok = false;
    tc_fence_after();
    batch1(0);  // its commit also covers C B^T
  }

  const int i = r;  // this thread's row (token) in the mask pass, and its token j in the epilogue
  const bool tok_ok = i < len;
  const int si = tok_ok ? sq[i] : -2;
  for (int hh = 0; hh < hpg; ++hh) {
    const int buf = hh & 1, h = h_first + hh;
    const long long bh = bh0 + hh;
    const uint8_t* sX = sXb + buf * kTok;
    const uint8_t* sY = sYb + buf * kTok;
    const float* l2 = l2q + buf * p.Q;
    const float* dtv = dtq + buf * p.Q;
    // scalars of head hh+1: loaded now, stored into the other slot (last read
    // by head hh-1) before this iteration's first barrier after the epilogue
    const bool pre = hh + 1 < hpg && tid < p.Q;
    float nl = 0.0f, nd = 0.0f;
    if (pre) {
      nl = f.lcs[(bh + 1) * p.Lp + t0 + tid];
      nd = f.dte[(bh + 1) * p.Lp + t0 + tid];
    }
    if (!mbar_wait(&bar[1 + buf], (hh >> 1) & 1)) ok = false;  // x, dy of head hh
    if (!wait_mma(&bar[4], ph_m1)) ok = false;                 // batch 1 of head hh
    if (tid == 0 && hh + 1 < hpg) issue_sh(hh + 1);            // dS, H have been consumed
    const float li2 = tok_ok ? l2[i] : 0.0f;
    // ---- mask pass: row i, columns 32 wg .. 32 wg + 31
    {
      float racc = 0.0f;
      for (int q = wg * 2; q < wg * 2 + 2; ++q) {
        uint32_t pk[8] = {0, 0, 0, 0, 0, 0, 0, 0};
        float cr = 0.0f, cq = 0.0f;
        if (q * 16 <= wlane + 31 && q * 16 < len) {  // warp-uniform; else every entry is masked
          float cb[16], dm[16], rv[16], qv[16];
          tmem_ld16x2(tmem_addr(tCB, wlane, q * 16), tmem_addr(tDM, wlane, q * 16), cb, dm);
#pragma unroll
          for (int e = 0; e < 16; e += 2) {
            const int j = q * 16 + e;
            const float2 lj = *reinterpret_cast<const float2*>(l2 + j);
            const float2 dj = *reinterpret_cast<const float2*>(dtv + j);
            const bool v0 = tok_ok && j <= i && (one_seg || sq[j] == si);
            const bool v1 = tok_ok && j + 1 <= i && (one_seg || sq[j + 1] == si);
            const float2 E = make_float2(exp2f(v0 ? li2 - lj.x : -INFINITY), exp2f(v1 ? li2 - lj.y : -INFINITY));
            const float2 cbE = __fmul2_rn(make_float2(cb[e], cb[e + 1]), E);
            const float2 m = __fmul2_rn(cbE, dj);
            const float2 dm2 = make_float2(dm[e], dm[e + 1]);
            const float2 rr = __fmul2_rn(dm2, m);
            const float2 qq = __fmul2_rn(dm2, cbE);
            rv[e] = rr.x;
            rv[e + 1] = rr.y;
            qv[e] = qq.x;
            qv[e + 1] = qq.y;
            racc += rr.x;
            racc += rr.y;
            pk[e / 2] = pack2(m.x, m.y);
          }
          cr = colsum16(rv, lane);
          cq = colsum16(qv, lane);
        }
        uint8_t* blk = sA + (q / 4) * kTok;
        const uint32_t e0 = (q % 4) * 16;
        *reinterpret_cast<uint4*>(blk + swz128_off(i, e0)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
        *reinterpret_cast<uint4*>(blk + swz128_off(i, e0 + 8)) = make_uint4(pk[4], pk[5], pk[6], pk[7]);
        if ((lane & 1) == 0) {
          const int col = q * 16 + ((lane >> 4) & 1) * 8 + ((lane >> 3) & 1) * 4 + ((lane >> 2) & 1) * 2 +
                          ((lane >> 1) & 1);
          colR[wq * kRows + col] = cr;
          colQ[wq * kRows + col] = cq;
        }
      }
      rowR[wg * kRows + i] = racc;
    }
    {  // carry term of dl_i: cv_i e^{l_i} dy_i . Yc_i (headdim columns 16 wg .. 16 wg + 15)
      float yc[16];
      tmem_ld16(tmem_addr(tYC, wlane, wg * 16), yc);
      const uint4 a = *reinterpret_cast<const uint4*>(sY + swz128_off(i, wg * 16));
      const uint4 b = *reinterpret_cast<const uint4*>(sY + swz128_off(i, wg * 16 + 8));
      const uint32_t dy[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
      float s = 0.0f;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float2 d = unpack2(dy[e]);
        s += d.x * yc[2 * e] + d.y * yc[2 * e + 1];
      }
      carP[wg * kRows + i] = (tok_ok && si == s_in) ? exp2f(li2) * s : 0.0f;
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();  // the M tile is complete; dM and Yc have been read
    if (tid == 0) {
      tc_fence_after();
      for (int ks = 0; ks < kRows / 16; ++ks) {  // dX = M^T dy (M = j, N = 64, K = tokens i)
        const uint64_t da = smem_desc(smem_u32(sA) + ks * 16 * 128, kTok, 1024, kSwz128);
        mma_bf16(tDX, da, mndesc_rows(sY, ks), id64t, ks > 0);
      }
      mma_commit(&bar[5]);
      if (hh + 1 < hpg) {  // batch 1 of the next head runs under this head's epilogue
        if (!mbar_wait(&bar[1 + (buf ^ 1)], ((hh + 1) >> 1) & 1)) ok = false;
        if (!mbar_wait(&bar[3], (hh + 1) & 1)) ok = false;
        tc_fence_after();
        batch1(hh + 1);
      }
    }
    // dl and ddt_eff partial sums of this head (token t = r, warpgroup 0)
    float dl_t = 0.0f, dd_t = 0.0f;
    if (wg == 0) {
      const int t = r;
      dl_t = ((rowR[t] + rowR[kRows + t]) + (rowR[2 * kRows + t] + rowR[3 * kRows + t])) +
             ((carP[t] + carP[kRows + t]) + (carP[2 * kRows + t] + carP[3 * kRows + t])) -
             ((colR[t] + colR[kRows + t]) + (colR[2 * kRows + t] + colR[3 * kRows + t]));
      dd_t = (colQ[t] + colQ[kRows + t]) + (colQ[2 * kRows + t] + colQ[3 * kRows + t]);
    }
    if (!wait_mma(&bar[5], ph_m2)) ok = false;  // dX of head hh
    // ---- epilogue: token j = r, headdim columns 16 wg .. 16 wg + 15
    {
      const int j = r;
      const float w = (tok_ok && sq[j] == s_last) ? exp2f(l2[len - 1] - l2[j]) : 0.0f;
      const float u = w * (tok_ok ? dtv[j] : 0.0f);
      const float Dh = f.D[h];
      float du = 0.0f, dyx = 0.0f;
      __nv_bfloat16* dx = static_cast<__nv_bfloat16*>(f.dx);
      const long long xrow = (((long long)bi * p.L + t0 + j) * p.H + h) * 64;
      const int q = wg;
      float a[16], s[16];
      tmem_ld16x2(tmem_addr(tDX, wlane, q * 16), tmem_addr(tDXS + buf * 64, wlane, q * 16), a, s);
      const uint4 x0 = *reinterpret_cast<const uint4*>(sX + swz128_off(j, q * 16));
      const uint4 x1 = *reinterpret_cast<const uint4*>(sX + swz128_off(j, q * 16 + 8));
      const uint4 y0 = *reinterpret_cast<const uint4*>(sY + swz128_off(j, q * 16));
      const uint4 y1 = *reinterpret_cast<const uint4*>(sY + swz128_off(j, q * 16 + 8));
      const uint32_t xs[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
      const uint32_t ys[8] = {y0.x, y0.y, y0.z, y0.w, y1.x, y1.y, y1.z, y1.w};
      uint32_t o[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float2 xv = unpack2(xs[e]), yv = unpack2(ys[e]);
        du += xv.x * s[2 * e] + xv.y * s[2 * e + 1];
        dyx += xv.x * yv.x + xv.y * yv.y;
        o[e] = pack2(a[2 * e] + u * s[2 * e] + Dh * yv.x, a[2 * e + 1] + u * s[2 * e + 1] + Dh * yv.y);
      }
      if (tok_ok) {
        uint4* dst = reinterpret_cast<uint4*>(dx + xrow + q * 16);
        dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
        dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
      }
      duP[wg * kRows + j] = du;
      dyxP[wg * kRows + j] = tok_ok ? dyx : 0.0f;
      if (pre) {
        l2q[(buf ^ 1) * p.Q + tid] = nl * kLog2e;
        dtq[(buf ^ 1) * p.Q + tid] = nd;
      }
      __syncthreads();
      if (wg == 0) {
        const float du_t = (duP[j] + duP[kRows + j]) + (duP[2 * kRows + j] + duP[3 * kRows + j]);
        float udu = 0.0f;
        if (tok_ok) {
          dd_t += w * du_t;
          dl_t -= u * du_t;
          udu = u * du_t;
          f.ddte[bh * p.Lp + t0 + j] = dd_t;
          f.dl[bh * p.Lp + t0 + j] = dl_t;
        }
        udu = warp_sum(udu);
        if (lane == 0) red[wq] = udu;
      } else if (wg == 1) {
        float v = (dyxP[j] + dyxP[kRows + j]) + (dyxP[2 * kRows + j] + dyxP[3 * kRows + j]);
        v = warp_sum(v);
        if (lane == 0) red[4 + wq] = v;
      }
    }
    tc_fence_before();
    __syncthreads();  // TMEM dX and the shared partials are reused by the next head
    if (tid == 0) {
      f.udu[bh * p.nc + c] = (red[0] + red[1]) + (red[2] + red[3]);
      f.pdD[((long long)bi * p.nc + c) * p.H + h] = (red[4] + red[5]) + (red[6] + red[7]);
      if (hh + 2 < hpg) issue_xy(hh + 2);  // this head's x, dy buffer is free
    }
  }
  if (!ok) atomicOr(&f.hdr->status, kDevTimeout);
  tc_fence_before();
  __syncthreads();
  if (tid < 32) tmem_dealloc(tm, 512);
}


// dB, dC of one chunk for one group (chunk <= 128): one CTA (512 threads) per
// (chunk, group, batch row) accumulates, in tensor memory and in fixed head
// order,
//   dC = sum_h [ dCB_h B + diag(cv e^{l_h}) dy_h H_h ],
//   dB = sum_h [ dCB_h^T C + diag(u_h) x_h dS_h ],   dCB_h = dM_h o E_h o dt_h.
// Per head: dM = dy x^T is issued one head ahead; once it has run, the x and
// dy tiles are scaled by their row factors in place and the carry and state
// MMAs are issued; meanwhile the 16 warps form dCB (thread = row i) as a bf16
// tile that is the K-major A of dCB B and the MN-major A of dCB^T C.
__global__ void __launch_bounds__(kThr, 1) chunk_bwd_dbc_group_tc_kernel(Plan p, Bufs f,
                                                                        const __grid_constant__ CUtensorMap tmX,
                                                                        const __grid_constant__ CUtensorMap tmY,
                                                                        const __grid_constant__ CUtensorMap tmB,
                                                                        const __grid_constant__ CUtensorMap tmC,
                                                                        const __grid_constant__ CUtensorMap tmS,
                                                                        const __grid_constant__ CUtensorMap tmH) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const GTiles T = gtiles(p.N, p.Q);
  uint8_t* sB = sm + T.offB;
  uint8_t* sC = sm + T.offC;
  uint8_t* sA = sm + T.offA;  // the dCB tile
  uint8_t* sXb = sm + T.offX;
  uint8_t* sYb = sm + T.offY;
  uint8_t* sS = sm + T.offS;
  uint8_t* sH = sm + T.offH;
  float* l2q = reinterpret_cast<float*>(sm + T.offF);  // [2 slots][Q]
  float* dtq = l2q + 2 * p.Q;                         // [2 slots][Q]
  int* sq = reinterpret_cast<int*>(dtq + 2 * p.Q);    // [Q]
  uint64_t* bar = reinterpret_cast<uint64_t*>(sq + p.Q + 24 * kRows + 8);  // ld_bc, ld_xy[2], ld_sh, dm, cs, dbc
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + 7);

  const int c = blockIdx.x, g = blockIdx.y, bi = blockIdx.z;
  const int tid = threadIdx.x;
  const int wg = tid >> 7, r = tid & 127, wq = (tid >> 5) & 3;
  const int wlane = wq * 32;
  const int t0 = c * p.Q, len = min(p.Q, p.L - t0);
  const int hpg = p.hpg, h_first = g * hpg;
  const long long bh0 = (long long)bi * p.H + h_first;

  for (int t = tid; t < p.Q; t += kThr) sq[t] = t < len ? seg_of(p, f, bi, (long long)t0 + t) : -1;
  if (tid < p.Q) {
    l2q[tid] = f.lcs[bh0 * p.Lp + t0 + tid] * kLog2e;
    dtq[tid] = f.dte[bh0 * p.Lp + t0 + tid];
  }
  zero_padding(T, sXb, sYb, sB, sC, tid);  // B and C are contracted over tokens here
  if (tid == 0) {
    for (int k = 0; k < 7; ++k) mbar_init(&bar[k], 1);
    mbar_fence_init();
  }
  if (tid < 32) tmem_alloc(tmem_slot, 512);
  fence_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tm = *tmem_slot;
  const uint32_t tDC = tm, tDB = tm + 128, tDM = tm + 256;
  const int s_in = seg_in_of(p, f, bi, c);
  const int s_last = sq[len - 1];
  const bool one_seg = sq[0] == s_last;
  bool ok = true;
  uint32_t ph_dm = 0, ph_dbc = 0;
  const uint32_t tok_bytes = (uint32_t)T.rows * 128u;
  const uint32_t c_bytes = (uint32_t)T.ncb * T.rows * T.cw;
  const uint32_t s_bytes = (uint32_t)p.N * 128u;
  const uint32_t idNk = idesc_bf16(128, p.N, 0, 0), idNmn = idesc_bf16(128, p.N, 0, 1);
  const uint32_t idNa_mn = idesc_bf16(128, p.N, 1, 1), id128 = idesc_bf16(128, 128, 0, 0);

  auto issue_xy = [&](int hh) {
    const int buf = hh & 1, h = h_first + hh;
    mbar_expect_tx(&bar[1 + buf], 2 * tok_bytes);
    tma_load_4d(sXb + buf * kTok, &tmX, &bar[1 + buf], 0, h, t0, bi);
    tma_load_4d(sYb + buf * kTok, &tmY, &bar[1 + buf], 0, h, t0, bi);
  };
  auto issue_sh = [&](int hh) {
    const int h = h_first + hh;
    mbar_expect_tx(&bar[3], 2 * s_bytes);
    tma_load_4d(sS, &tmS, &bar[3], 0, 0, c, bi * p.H + h);
    tma_load_4d(sH, &tmH, &bar[3], 0, 0, c, bi * p.H + h);
  };
  auto kdesc_tok = [&](const uint8_t* t, int ks) { return smem_desc(smem_u32(t) + ks * 32, 16, 1024, kSwz128); };
  auto mndesc_c = [&](const uint8_t* t, int ks) {  // B/C tile as MN-major (N = d_state), K = tokens
    return smem_desc(smem_u32(t) + ks * 16 * T.cw, T.cblk, 8 * T.cw, T.cswz);
  };
  auto issue_dm = [&](int hh) {  // dM = dy x^T of head hh (M = i, N = j, K = headdim)
    const int buf = hh & 1;
    for (int ks = 0; ks < 4; ++ks)
      mma_bf16(tDM, kdesc_tok(sYb + buf * kTok, ks), kdesc_tok(sXb + buf * kTok, ks), id128, ks > 0);
    mma_commit(&bar[4]);
  };

  if (tid == 0) {
    mbar_expect_tx(&bar[0], 2 * c_bytes);
    for (int q = 0; q < T.ncb; ++q) {
      tma_load_4d(sB + q * T.cblk, &tmB, &bar[0], q * 64, g, t0, bi);
      tma_load_4d(sC + q * T.cblk, &tmC, &bar[0], q * 64, g, t0, bi);
    }
    issue_xy(0);
    if (hpg > 1) issue_xy(1);
    issue_sh(0);
    if (!mbar_wait(&bar[1], 0)) ok = false;
    tc_fence_after();
    issue_dm(0);
  }

  const int i = r;
  const bool tok_ok = i < len;
  const int si = tok_ok ? sq[i] : -2;
  for (int hh = 0; hh < hpg; ++hh) {
    const int buf = hh & 1;
    uint8_t* sX = sXb + buf * kTok;
    uint8_t* sY = sYb + buf * kTok;
    const float* l2 = l2q + buf * p.Q;
    const float* dtv = dtq + buf * p.Q;
    const bool pre = hh + 1 < hpg && tid < p.Q;
    float nl = 0.0f, nd = 0.0f;
    if (pre) {
      const long long bhn = bh0 + hh + 1;
      nl = f.lcs[bhn * p.Lp + t0 + tid];
      nd = f.dte[bhn * p.Lp + t0 + tid];
    }
    if (!mbar_wait(&bar[1 + buf], (hh >> 1) & 1)) ok = false;  // x, dy of head hh
    if (!wait_mma(&bar[4], ph_dm)) ok = false;                 // dM of head hh has read them
    // row scaling in place: warpgroups 0, 1 -> cv e^{l} dy (rows i), 2, 3 -> u x (rows j)
    {
      const int t = r;
      const bool v = t < len;
      float sc;
      uint8_t* tile;
      if (wg < 2) {
        sc = (v && sq[t] == s_in) ? exp2f(l2[t]) : 0.0f;
        tile = sY;
      } else {
        sc = (v && sq[t] == s_last) ? exp2f(l2[len - 1] - l2[t]) * dtv[t] : 0.0f;
        tile = sX;
      }
      const float2 sc2 = make_float2(sc, sc);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint32_t off = swz128_off(t, (wg & 1) * 32 + k * 8);
        const uint4 w4 = *reinterpret_cast<const uint4*>(tile + off);
        const uint32_t a[4] = {w4.x, w4.y, w4.z, w4.w};
        uint32_t o[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 x2 = __fmul2_rn(unpack2(a[e]), sc2);
          o[e] = pack2(x2.x, x2.y);
        }
        *reinterpret_cast<uint4*>(tile + off) = make_uint4(o[0], o[1], o[2], o[3]);
      }
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    if (tid == 0) {  // carry and state: dC += (scaled dy) H, dB += (scaled x) dS  (K = headdim)
      if (!mbar_wait(&bar[3], hh & 1)) ok = false;  // dS, H of head hh
      tc_fence_after();
      for (int ks = 0; ks < 4; ++ks) {
        mma_bf16(tDC, kdesc_tok(sY, ks), kdesc_tok(sH, ks), idNk, (hh > 0 || ks > 0) ? 1u : 0u);
        mma_bf16(tDB, kdesc_tok(sX, ks), kdesc_tok(sS, ks), idNk, (hh > 0 || ks > 0) ? 1u : 0u);
      }
      mma_commit(&bar[5]);
    }
    // dCB = dM o E o dt (row i, columns 32 wg .. 32 wg + 31); the dB/dC MMAs
    // of head hh-1 must have read the previous dCB tile first
    if (hh > 0 && !wait_mma(&bar[6], ph_dbc)) ok = false;
    {
      const float li2 = tok_ok ? l2[i] : 0.0f;
      for (int q = wg * 2; q < wg * 2 + 2; ++q) {
        uint32_t pk[8] = {0, 0, 0, 0, 0, 0, 0, 0};
        if (q * 16 <= wlane + 31 && q * 16 < len) {  // warp-uniform; else every entry is masked
          float dm[16];
          tmem_ld16(tmem_addr(tDM, wlane, q * 16), dm);
#pragma unroll
          for (int e = 0; e < 16; e += 2) {
            const int j = q * 16 + e;
            const float2 lj = *reinterpret_cast<const float2*>(l2 + j);
            const float2 dj = *reinterpret_cast<const float2*>(dtv + j);
            const bool v0 = tok_ok && j <= i && (one_seg || sq[j] == si);
            const bool v1 = tok_ok && j + 1 <= i && (one_seg || sq[j + 1] == si);
            const float2 E = make_float2(exp2f(v0 ? li2 - lj.x : -INFINITY), exp2f(v1 ? li2 - lj.y : -INFINITY));
            const float2 v2 = __fmul2_rn(__fmul2_rn(make_float2(dm[e], dm[e + 1]), E), dj);
            pk[e / 2] = pack2(v2.x, v2.y);
          }
        }
        uint8_t* blk = sA + (q / 4) * kTok;
        const uint32_t e0 = (q % 4) * 16;
        *reinterpret_cast<uint4*>(blk + swz128_off(i, e0)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
        *reinterpret_cast<uint4*>(blk + swz128_off(i, e0 + 8)) = make_uint4(pk[4], pk[5], pk[6], pk[7]);
      }
    }
    if (pre) {  // the other slot was last read by head hh-1
      l2q[(buf ^ 1) * p.Q + tid] = nl * kLog2e;
      dtq[(buf ^ 1) * p.Q + tid] = nd;
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    if (tid == 0) {
      tc_fence_after();
      if (hh + 1 < hpg) {  // dM of the next head first: the tensor core has the dB/dC work to hide it
        if (!mbar_wait(&bar[1 + (buf ^ 1)], ((hh + 1) >> 1) & 1)) ok = false;
        tc_fence_after();
        issue_dm(hh + 1);
      }
      if (hh == 0 && !mbar_wait(&bar[0], 0)) ok = false;  // B, C
      tc_fence_after();
      // dC += dCB B (A K-major, K = j);  dB += dCB^T C (A MN-major, K = i)
      for (int ks = 0; ks < kRows / 16; ++ks) {
        const uint64_t ak = smem_desc(smem_u32(sA) + (ks / 4) * kTok + (ks % 4) * 32, 16, 1024, kSwz128);
        const uint64_t am = smem_desc(smem_u32(sA) + ks * 16 * 128, kTok, 1024, kSwz128);
        mma_bf16(tDC, ak, mndesc_c(sB, ks), idNmn, 1u);
        mma_bf16(tDB, am, mndesc_c(sC, ks), idNa_mn, 1u);
      }
      mma_commit(&bar[6]);
      // the carry and state MMAs of this head are done long since: release
      // dS, H and this head's x, dy buffer to the next loads
      if (!mbar_wait(&bar[5], hh & 1)) ok = false;
      if (hh + 1 < hpg) issue_sh(hh + 1);
      if (hh + 2 < hpg) issue_xy(hh + 2);
    }
  }
  if (!wait_mma(&bar[6], ph_dbc)) ok = false;  // the last head's dB/dC MMAs
  // epilogue: rows of dB and dC (thread = token t; d_state columns 16 q, q = wg mod 4)
  {
    const int t = r;
    const bool v = t < len;
    __nv_bfloat16* dB = static_cast<__nv_bfloat16*>(f.dB);
    __nv_bfloat16* dC = static_cast<__nv_bfloat16*>(f.dC);
    const long long row = (((long long)bi * p.L + t0 + t) * p.G + g) * p.N;
    const int nq = p.N / 16;
    for (int q = wg; q < nq; q += 4) {
      float vb[16], vc[16];
      tmem_ld16x2(tmem_addr(tDB, wlane, q * 16), tmem_addr(tDC, wlane, q * 16), vb, vc);
      if (v) {
        uint4* ob = reinterpret_cast<uint4*>(dB + row + q * 16);
        uint4* oc = reinterpret_cast<uint4*>(dC + row + q * 16);
        ob[0] = make_uint4(pack2(vb[0], vb[1]), pack2(vb[2], vb[3]), pack2(vb[4], vb[5]), pack2(vb[6], vb[7]));
        ob[1] = make_uint4(pack2(vb[8], vb[9]), pack2(vb[10], vb[11]), pack2(vb[12], vb[13]), pack2(vb[14], vb[15]));
        oc[0] = make_uint4(pack2(vc[0], vc[1]), pack2(vc[2], vc[3]), pack2(vc[4], vc[5]), pack2(vc[6], vc[7]));
        oc[1] = make_uint4(pack2(vc[8], vc[9]), pack2(vc[10], vc[11]), pack2(vc[12], vc[13]), pack2(vc[14], vc[15]));
      }
    }
  }
  if (!ok) atomicOr(&f.hdr->status, kDevTimeout);
  tc_fence_before();
  __syncthreads();
  if (tid < 32) tmem_dealloc(tm, 512);
}

}  // namespace

bool chunk_bwd_group_tc_supported(const Plan& p) {
  return p.dtype == SSD_BF16 && p.P == 64 && (p.Q == 64 || p.Q == 128) &&
         (p.N == 16 || p.N == 32 || p.N == 64 || p.N == 128);
}

namespace {
bool group_maps(const Plan& p, const Bufs& f, CUtensorMap* X, CUtensorMap* Y, CUtensorMap* B, CUtensorMap* C,
                CUtensorMap* S, CUtensorMap* H) {
  const GTiles T = gtiles(p.N, p.Q);
  const uint32_t rows = (uint32_t)T.rows;
  const uint64_t dbc[4] = {(uint64_t)p.N, (uint64_t)p.G, (uint64_t)p.L, (uint64_t)p.b};
  const uint64_t sbc[3] = {(uint64_t)p.N * 2, (uint64_t)p.G * p.N * 2, (uint64_t)p.L * p.G * p.N * 2};
  const uint32_t bbc[4] = {(uint32_t)(T.cw / 2), 1, rows, 1};
  const uint64_t dxx[4] = {64, (uint64_t)p.H, (uint64_t)p.L, (uint64_t)p.b};
  const uint64_t sxx[3] = {128, (uint64_t)p.H * 128, (uint64_t)p.L * p.H * 128};
  const uint32_t bxx[4] = {64, 1, rows, 1};
  const uint64_t ds[4] = {64, (uint64_t)p.N, (uint64_t)p.nc, (uint64_t)p.b * p.H};
  const uint64_t ss[3] = {128, (uint64_t)p.N * 128, (uint64_t)p.nc * p.N * 128};
  const uint32_t bs[4] = {64, (uint32_t)p.N, 1, 1};
  return encode_tmap_bf16_4d(X, f.x, dxx, sxx, bxx, 128) && encode_tmap_bf16_4d(Y, f.dy, dxx, sxx, bxx, 128) &&
         encode_tmap_bf16_4d(B, f.B, dbc, sbc, bbc, T.cw) && encode_tmap_bf16_4d(C, f.C, dbc, sbc, bbc, T.cw) &&
         encode_tmap_bf16_4d(S, f.dS, ds, ss, bs, 128) && encode_tmap_bf16_4d(H, f.Hin, ds, ss, bs, 128);
}
}  // namespace

cudaError_t launch_chunk_bwd_dbc_group_tc(const Plan& p, const Bufs& f, cudaStream_t s) {
  set_kernel_name("chunk_bwd_dbc_tc");
  const GTiles T = gtiles(p.N, p.Q);
  CUtensorMap X, Y, B, C, S, H;
  if (!group_maps(p, f, &X, &Y, &B, &C, &S, &H)) return cudaErrorInvalidValue;
  const size_t smem = group_smem_bytes(T, p.Q);
  cudaError_t e = cudaFuncSetAttribute(chunk_bwd_dbc_group_tc_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  chunk_bwd_dbc_group_tc_kernel<<<dim3(p.nc, p.G, p.b), kThr, smem, s>>>(p, f, X, Y, B, C, S, H);
  return cudaGetLastError();
}

cudaError_t launch_chunk_bwd_group_tc(const Plan& p, const Bufs& f, cudaStream_t s) {
  set_kernel_name("chunk_bwd_tc");
  const GTiles T = gtiles(p.N, p.Q);
  CUtensorMap X, Y, B, C, S, H;
  if (!group_maps(p, f, &X, &Y, &B, &C, &S, &H)) return cudaErrorInvalidValue;
  const size_t smem = group_smem_bytes(T, p.Q);
  cudaError_t e = cudaFuncSetAttribute(chunk_bwd_group_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  chunk_bwd_group_tc_kernel<<<dim3(p.nc, p.G, p.b), kThr, smem, s>>>(p, f, X, Y, B, C, S, H);
  return cudaGetLastError();
}

cudaError_t launch_chunk_bwd_pair_tc(const Plan& p, const Bufs& f, cudaStream_t s);
cudaError_t launch_chunk_bwd_dbc_tc(const Plan& p, const Bufs& f, cudaStream_t s);
bool chunk_bwd_pair_tc_supported(const Plan& p);

bool chunk_bwd_tc_supported(const Plan& p) {
  return chunk_bwd_group_tc_supported(p) || chunk_bwd_pair_tc_supported(p);
}

// Token gradients (per head) then dB, dC (per group).  Chunks of up to 128
// tokens use the group kernel; 256-token chunks the per-head block-pair kernel.
cudaError_t launch_chunk_bwd_tc(const Plan& p, const Bufs& f, cudaStream_t s) {
  cudaError_t e = chunk_bwd_group_tc_supported(p) ? launch_chunk_bwd_group_tc(p, f, s)
                                                  : launch_chunk_bwd_pair_tc(p, f, s);
  if (e != cudaSuccess) return e;
  prof_after(s);  // the entry point brackets one launch; time the second kernel on its own
  prof_before(s);
  return chunk_bwd_group_tc_supported(p) ? launch_chunk_bwd_dbc_group_tc(p, f, s) : launch_chunk_bwd_dbc_tc(p, f, s);
}

}  // namespace ssd
