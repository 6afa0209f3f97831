// k_chunk_bwd_tok_tc.cu -- per-head token gradients of one 128-token chunk for
// all heads of one group, on the 5th-generation tensor cores.
//
// Notation (chunk c, head h, chunk-local tokens i, j):
//   E_ij  = exp(l_i - l_j) [j <= i, seg_i = seg_j],   M'_ij = (C_i . B_j) E_ij,
//   M_ij  = M'_ij dt_j (the chunk-output operator),   dM_ij = dy_i . x_j,
//   u_j   = w_j dt_j,  w_j = sv_j exp(l_last - l_j),  dS = dL/dS_c,  H = carry-in state.
// Per head the layer's reverse mode needs
//   dx_j      = sum_i M_ij dy_i + u_j dS B_j + D_h dy_j
//   ddt_eff_j = sum_i dM_ij M'_ij + w_j (x_j . dS B_j)
//   dl_t      = sum_j dM_tj M_tj - sum_i dM_it M_it + cv_t e^{l_t} dy_t . (H C_t) - u_t (x_t . dS B_t)
// and the per-chunk sums of u_j (x_j . dS B_j) and dy . x.  Every sum over
// i or j factors through a product the tensor core forms (dM_ij = dy_i . x_j):
//   Z = M^T dY:  sum_i M_ij dy_i = Z_j,   sum_i dM_it M_it = x_t . Z_t,
//                sum_i dM_ij M'_ij = (x_j . Z_j) / dt_j
//   W = M X:     sum_j dM_tj M_tj = dy_t . W_t
// so the element-wise pass only forms the bf16 tile M (no dM product, no
// column sums), and every gradient is a 64-long dot product of rows the
// thread of token t already holds.  The row and column sums of dM o M come
// from the same bf16 tile, so dl's two sums -- whose difference is summed
// again over the chunk by the parameter gradients -- carry the same
// rounding and cancel as exactly as they would in fp32.  (Dividing by dt_j
// is guarded: below 1e-30 the term is dropped, where it is multiplied by
// sigmoid(dt + dt_bias) ~ dt_j < 1e-30 on its way to ddt.)  (Page "B200 Helion Mamba-2"
// (aitrends.kr/articles/109906), section "Helion based B200 kernel redesign":
// TMA, TMEM and warp specialisation on Blackwell; the derivation of the
// reverse mode is this library's, from the recurrence.)
//
// A work unit is one (chunk, group, batch row); a persistent CTA per SM takes
// units blockIdx.x, blockIdx.x + gridDim.x, ... and walks the heads of its
// units as one sequence, so the copies and products of a unit's first head
// overlap the last heads of the unit before.  16 compute warps (warp w reads
// TMEM lane quarter w % 4) and two control warps, one lane of each issuing:
//   control A: the B, C, dS, H copies, C B^T once per unit, per head
//     dXs = B dS^T and Yc = C H^T (as soon as the previous head's epilogue
//     has read them);
//   control B: the x, dy copies, per head Z = M^T dY and W = M X into a
//     double-buffered pair, the dx stores;
//   compute, per head: the M tile (units strictly below a row block's
//     diagonal block use exp(l_i - l_r) exp(l_r - l_j) dt_j, l_r the block's
//     first row, both exponentials <= 1, the second from a per-warp table
//     of the warp's columns),
//     then the epilogue of the previous head while the tensor core forms Z, W
//     of this one.
// Per-token results leave through fixed-order folds of the four warpgroups'
// partial dot products; the per-chunk sums through fixed warp butterflies.
#include "ssd_internal.cuh"
#include "tc_common.cuh"
#include "tma_host.h"

namespace ssd {

namespace {

using namespace tc;

constexpr int kQ = 128;
constexpr int kCompute = 512;
constexpr int kThr = kCompute + 64;
constexpr unsigned kFull = 0xffffffffu;
constexpr uint32_t kTok = kQ * 128u;  // one (128 tokens x 64) bf16 tile

__host__ __device__ inline uint32_t r1024(uint32_t v) { return (v + 1023u) & ~1023u; }

struct TokGeom {
  int cw, ncb;
  uint32_t cblk, cswz, cbytes, sbytes;
  uint32_t offB, offC, offA, offX, offY, offS, offH, offF;
};

__host__ __device__ inline TokGeom tok_geom(int N) {
  TokGeom t;
  t.cw = 2 * (N < 64 ? N : 64);
  t.ncb = N >= 64 ? N / 64 : 1;
  t.cblk = (uint32_t)kQ * t.cw;
  t.cswz = t.cw == 128 ? kSwz128 : (t.cw == 64 ? kSwz64 : kSwz32);
  t.cbytes = r1024(t.ncb * t.cblk);
  t.sbytes = r1024((uint32_t)N * 128u);
  t.offB = 0;
  t.offC = t.cbytes;
  t.offA = 2 * t.cbytes;       // M tile, 128 x 128 bf16 (two 64-column blocks)
  t.offX = t.offA + 2 * kTok;  // [2] x tiles
  t.offY = t.offX + 2 * kTok;  // [2] dy tiles
  t.offS = t.offY + 2 * kTok;  // dS tile
  t.offH = t.offS + t.sbytes;  // H tile
  t.offF = t.offH + t.sbytes;
  return t;
}

// floats after offF: l, dt [3 slots][Q]; segment ids [4 units][Q]; unit
// table [4][8]; a 32-entry factor table per compute warp [16][32];
// five partial arrays [4][Q]; per-warp sums [8]; then the barriers and the
// TMEM address
constexpr int kRingU = 4;  // units whose segment ids and coordinates are kept
constexpr int kFloats = 3 * kQ + 3 * kQ + kRingU * kQ + kRingU * 8 + 4 * kQ + 20 * kQ + 8;

__host__ __device__ inline size_t tok_smem_bytes(const TokGeom& T) {
  return 1024 + T.offF + (size_t)kFloats * 4 + 16 * 8 + 16;
}

__device__ __forceinline__ uint32_t pack2(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}
__device__ __forceinline__ float2 unpack2(uint32_t v) {
  return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&v));
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
  return v;
}
__device__ __forceinline__ void named_sync_compute() {
  asm volatile("bar.sync 1, %0;" ::"n"(kCompute) : "memory");
}

// One work unit: chunk c (tokens t0 .. t0 + len - 1) of batch row bi, group g
// (the launcher keeps the unit count below 2^31).
struct TokUnit {
  int c, g, bi, t0, len;
};
__device__ __forceinline__ TokUnit tok_unit(const Plan& p, uint32_t u) {
  TokUnit w;
  const uint32_t nc = (uint32_t)p.nc, G = (uint32_t)p.G;
  const uint32_t r = u / nc, bi = r / G;
  w.c = (int)(u - r * nc);
  w.g = (int)(r - bi * G);
  w.bi = (int)bi;
  w.t0 = w.c * kQ;
  w.len = min(kQ, p.L - w.t0);
  return w;
}
// Unit table entry (ints): c, g, bi, t0, len, segment id entering the unit.
enum { kUc = 0, kUg, kUbi, kUt0, kUlen, kUsin };

__global__ void __launch_bounds__(kThr, 1) chunk_bwd_tok_tc_kernel(Plan p, Bufs f,
                                                                 const __grid_constant__ CUtensorMap tmX,
                                                                 const __grid_constant__ CUtensorMap tmY,
                                                                 const __grid_constant__ CUtensorMap tmB,
                                                                 const __grid_constant__ CUtensorMap tmC,
                                                                 const __grid_constant__ CUtensorMap tmS,
                                                                 const __grid_constant__ CUtensorMap tmH,
                                                                 const __grid_constant__ CUtensorMap tmDX) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const TokGeom T = tok_geom(p.N);
  uint8_t* sB = sm + T.offB;
  uint8_t* sC = sm + T.offC;
  uint8_t* sA = sm + T.offA;
  uint8_t* sXb = sm + T.offX;
  uint8_t* sYb = sm + T.offY;
  uint8_t* sS = sm + T.offS;
  uint8_t* sH = sm + T.offH;
  float* lq = reinterpret_cast<float*>(sm + T.offF);  // [3][Q]
  float* dtq = lq + 3 * kQ;                           // [3][Q]
  int* sqr = reinterpret_cast<int*>(dtq + 3 * kQ);    // [kRingU][Q] segment ids
  int* utab = sqr + kRingU * kQ;                      // [kRingU][8] unit table
  float* wtab = reinterpret_cast<float*>(utab + kRingU * 8);  // [warp][32] exp(l_r - l_j) dt_j
  float* pZX = wtab + 4 * kQ;                         // [4 warpgroups][Q] x . Z
  float* pWY = pZX + 4 * kQ;                          // dy . W
  float* pDU = pWY + 4 * kQ;                          // x . dXs
  float* pCA = pDU + 4 * kQ;                          // dy . Yc
  float* pYX = pCA + 4 * kQ;                          // dy . x
  float* red = pYX + 4 * kQ;                          // [8]
  uint64_t* bar = reinterpret_cast<uint64_t*>(red + 8);
  uint64_t *b_bc = bar, *b_xy = bar + 1, *b_sh = bar + 3, *b_cb = bar + 4, *b_b1 = bar + 5, *b_mr = bar + 6,
           *b_b2 = bar + 7, *b_ed = bar + 9, *b_bf = bar + 11;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + 16);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int wg = (tid >> 7) & 3, r = tid & 127, wq = (tid >> 5) & 3;
  const int wlane = wq * 32;
  const int hpg = p.hpg;
  const uint32_t nunits_all = (uint32_t)p.nc * (uint32_t)p.G * (uint32_t)p.b;
  const int nunits = (int)((nunits_all - blockIdx.x + gridDim.x - 1) / gridDim.x);
  const int nh = nunits * hpg;  // heads this CTA walks, unit by unit
  auto unit_of = [&](int i) { return tok_unit(p, blockIdx.x + (uint32_t)i * gridDim.x); };
  const uint32_t c_bytes = (uint32_t)T.ncb * T.cblk;
  const uint32_t s_bytes = (uint32_t)p.N * 128u;
  // segment ids and table entry of unit i into ring slot i % kRingU
  // (threads 0 .. Q-1)
  auto fill_unit = [&](int i) {
    if (tid < kQ && i < nunits) {
      const TokUnit w = unit_of(i);
      const int slot = i % kRingU;
      sqr[slot * kQ + tid] = tid < w.len ? seg_of(p, f, w.bi, (long long)w.t0 + tid) : -1;
      if (tid == 0) {
        int* u = utab + slot * 8;
        u[kUc] = w.c;
        u[kUg] = w.g;
        u[kUbi] = w.bi;
        u[kUt0] = w.t0;
        u[kUlen] = w.len;
        u[kUsin] = seg_in_of(p, f, w.bi, w.c);
      }
    }
  };
  if (tid == kCompute) {
    // bc, xy[2], sh, cb, b1, mr (one arrival per compute warp), b2[2], ed[2]
    for (int k = 0; k < 11; ++k) mbar_init(&bar[k], bar + k == b_mr ? kCompute / 32 : 1);
    mbar_init(b_bf, kCompute / 32);                      // one arrival per compute warp
    mbar_fence_init();
  }
  fill_unit(0);
  fill_unit(1);
  if (tid < kQ && nh > 0) {  // scalars of the first head into slot 0
    const TokUnit w = unit_of(0);
    const long long bh = (long long)w.bi * p.H + w.g * hpg;
    lq[tid] = f.lcs[bh * p.Lp + w.t0 + tid];
    dtq[tid] = f.dte[bh * p.Lp + w.t0 + tid];
  }
  if (warp == 0) tmem_alloc(tmem_slot, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tm = *tmem_slot;
  // C B^T | [2] (Z | W) | dXs | Yc
  const uint32_t tCB = tm, tZW = tm + 128, tDXS = tm + 384, tYC = tm + 448;
  bool ok = true;
  auto wait = [&](uint64_t* b, uint32_t ph) { mbar_wait_flag(b, ph, ok); };

  if (warp >= kCompute / 32) {
    const int cw = warp - kCompute / 32;
    if (lane == 0 && nh > 0) {
      const uint32_t id128 = idesc_bf16(128, 128, 0, 0), id64 = idesc_bf16(128, 64, 0, 1);
      const uint32_t id64t = idesc_bf16(128, 64, 1, 1);
      // row width of the B/C tile is 32, 64 or 128 bytes: shifts, not divisions
      const uint32_t lcw = T.cw == 128 ? 7u : (T.cw == 64 ? 6u : 5u);
      auto kdesc_c = [&](const uint8_t* t, int ks) {  // K-major B/C tile, K = d_state
        const uint32_t kb = ((uint32_t)ks * 32u) >> lcw, kin = ((uint32_t)ks * 32u) & (T.cw - 1u);
        return smem_desc(smem_u32(t) + kb * T.cblk + kin, 16, 8 * T.cw, T.cswz);
      };
      auto mndesc_rows = [&](const uint8_t* t, int ks) {  // MN-major (64 wide), K along rows
        return smem_desc(smem_u32(t) + ks * 16 * 128, 16, 1024, kSwz128);
      };
      // copies of head hh of unit w into buffer buf, and its dx store
      auto issue_xy = [&](const TokUnit& w, int hh, int buf) {
        const int h = w.g * hpg + hh;
        mbar_expect_tx(&b_xy[buf], 2 * kTok);
        tma_load_4d(sXb + buf * kTok, &tmX, &b_xy[buf], 0, h, w.t0, w.bi);
        tma_load_4d(sYb + buf * kTok, &tmY, &b_xy[buf], 0, h, w.t0, w.bi);
      };
      auto store_dx = [&](const TokUnit& w, int hh, int buf) {
        tma_store_4d(&tmDX, sYb + buf * kTok, 0, w.g * hpg + hh, w.t0, w.bi);
        bulk_commit();
      };
      TokUnit uprev, ucur = unit_of(0), unext = unit_of(nunits > 1 ? 1 : 0);
      uprev = ucur;
      if (cw == 0) {
        // ---------------- control A: B, C, dS, H copies; C B^T; per head dXs and Yc ----------------
        auto issue_sh = [&](const TokUnit& w, int hh) {
          const int bhh = w.bi * p.H + w.g * hpg + hh;
          mbar_expect_tx(b_sh, 2 * s_bytes);
          tma_load_4d(sS, &tmS, b_sh, 0, 0, w.c, bhh);
          tma_load_4d(sH, &tmH, b_sh, 0, 0, w.c, bhh);
        };
        auto issue_bc = [&](const TokUnit& w) {
          mbar_expect_tx(b_bc, 2 * c_bytes);
          for (int q = 0; q < T.ncb; ++q) {
            tma_load_4d(sB + q * T.cblk, &tmB, b_bc, q * 64, w.g, w.t0, w.bi);
            tma_load_4d(sC + q * T.cblk, &tmC, b_bc, q * 64, w.g, w.t0, w.bi);
          }
        };
        issue_bc(ucur);
        issue_sh(ucur, 0);
        int i = 0, hh = 0;  // unit and head of k
        for (int k = 0; k < nh; ++k) {
          if (hh == 0) {
            if (k > 0) {
              ucur = unext;
              unext = unit_of(i + 1 < nunits ? i + 1 : i);
            }
            wait(b_bc, i & 1);
            // the mask pass of the previous unit's last head has read C B^T
            if (k > 0) wait(b_mr, (k - 1) & 1);
            tc_fence_after();
            for (int ks = 0; ks < p.N / 16; ++ks)  // C B^T (M = i, N = j, K = d_state), once per unit
              mma_bf16(tCB, kdesc_c(sC, ks), kdesc_c(sB, ks), id128, ks > 0);
            mma_commit(b_cb);
          }
          wait(b_sh, k & 1);
          if (k >= 1) wait(b_bf, (k - 1) & 1);  // the previous head's epilogue has read dXs, Yc
          tc_fence_after();
          for (int ks = 0; ks < p.N / 16; ++ks) {
            mma_bf16(tDXS, kdesc_c(sB, ks), mndesc_rows(sS, ks), id64, ks > 0);
            mma_bf16(tYC, kdesc_c(sC, ks), mndesc_rows(sH, ks), id64, ks > 0);
          }
          mma_commit(b_b1);
          if (k + 1 < nh) {
            wait(b_b1, k & 1);  // dS, H read; the unit's B, C too if this was its last head
            if (hh + 1 == hpg) {
              issue_bc(unext);
              issue_sh(unext, 0);
            } else {
              issue_sh(ucur, hh + 1);
            }
          }
          if (++hh == hpg) {
            hh = 0;
            ++i;
          }
        }
      } else {
        // ---------------- control B: x, dy copies; per head Z = M^T dY, W = M X; dx stores ----------------
        issue_xy(ucur, 0, 0);
        if (nh > 1) {
          if (hpg > 1) issue_xy(ucur, 1, 1);
          else issue_xy(unext, 0, 1);
        }
        int i = 0, hh = 0;  // unit and head of k
        for (int k = 0; k < nh; ++k) {
          if (hh == 0 && k > 0) {
            uprev = ucur;
            ucur = unext;
            unext = unit_of(i + 1 < nunits ? i + 1 : i);
          }
          // M of head k written; the pair k & 1 was read by the epilogue of
          // head k-2, which the compute warps finished first; x, dy of head
          // k landed (the mask pass does not read them)
          wait(b_mr, k & 1);
          wait(&b_xy[k & 1], (k >> 1) & 1);
          tc_fence_after();
          const uint32_t tz = tZW + (k & 1) * 128, tw = tz + 64;
          const uint8_t* sY = sYb + (k & 1) * kTok;
          const uint8_t* sX = sXb + (k & 1) * kTok;
          for (int ks = 0; ks < kQ / 16; ++ks) {
            const uint64_t am = smem_desc(smem_u32(sA) + ks * 16 * 128, kTok, 1024, kSwz128);   // M^T
            const uint64_t ak = smem_desc(smem_u32(sA) + (ks / 4) * kTok + (ks % 4) * 32, 16, 1024, kSwz128);
            mma_bf16(tz, am, mndesc_rows(sY, ks), id64t, ks > 0);
            mma_bf16(tw, ak, mndesc_rows(sX, ks), id64, ks > 0);
          }
          mma_commit(&b_b2[k & 1]);
          if (k >= 1) {
            // the previous head's epilogue left its dx in its dy tile: store
            // it, then refill that buffer with the next head once the store
            // has read it
            wait(&b_ed[(k - 1) & 1], ((k - 1) >> 1) & 1);
            if (hh == 0) store_dx(uprev, hpg - 1, (k - 1) & 1);
            else store_dx(ucur, hh - 1, (k - 1) & 1);
            if (k + 1 < nh) {
              bulk_wait_read<0>();
              if (hh + 1 == hpg) issue_xy(unext, 0, (k + 1) & 1);
              else issue_xy(ucur, hh + 1, (k + 1) & 1);
            }
          }
          if (++hh == hpg) {
            hh = 0;
            ++i;
          }
        }
        wait(&b_ed[(nh - 1) & 1], ((nh - 1) >> 1) & 1);  // the last head's dx
        store_dx(ucur, hpg - 1, (nh - 1) & 1);
        bulk_wait_all();
      }
    }
  } else if (nh > 0) {
    // ---------------- 16 compute warps ----------------
    const int i_row = wlane + lane;  // row of this thread in the mask pass
    // upper-triangle 16-column units of the M tile: zero once
    for (int q = 2 * wq + 2 + wg; q < 8; q += 4) {
      uint8_t* blk = sA + (q >> 2) * kTok;
      const uint32_t e0 = (q & 3) * 16;
      *reinterpret_cast<uint4*>(blk + swz128_off(i_row, e0)) = make_uint4(0, 0, 0, 0);
      *reinterpret_cast<uint4*>(blk + swz128_off(i_row, e0 + 8)) = make_uint4(0, 0, 0, 0);
    }
    named_sync_compute();

    // ---- M tile of head k (head hh of unit iu)
    auto mask_pass = [&](int k, int iu, int hh) {
      const int us = iu % kRingU;
      const int* ut = utab + us * 8;
      const int* sq = sqr + us * kQ;
      const int slot = k % 3;
      const float* lb = lq + slot * kQ;
      const float* db = dtq + slot * kQ;
      if (hh == 0) {
        // table entries of the unit after next: its ring slot was last read by
        // the epilogues of the unit two back, all done
        fill_unit(iu + 2);
        wait(b_cb, iu & 1);
        tc_fence_after();
      }
      const int iu_n = hh + 1 == hpg ? iu + 1 : iu, hh_n = hh + 1 == hpg ? 0 : hh + 1;
      if (k + 1 < nh && tid < kQ) {  // scalars of head k+1 (slot last read by head k-2)
        const int* un = utab + (iu_n % kRingU) * 8;
        const long long bhn = (long long)un[kUbi] * p.H + un[kUg] * hpg + hh_n;
        const int sn = (k + 1) % 3;
        cp_async4(lq + sn * kQ + tid, f.lcs + bhn * p.Lp + un[kUt0] + tid);
        cp_async4(dtq + sn * kQ + tid, f.dte + bhn * p.Lp + un[kUt0] + tid);
      }
      cp_async_commit();
      if (k >= 1) {  // Z, W of head k-1 done: M may be rewritten
        wait(&b_b2[(k - 1) & 1], ((k - 1) >> 1) & 1);
        tc_fence_after();
      }
      const int len = ut[kUlen];
      const int s_last = sq[len - 1];
      const bool one_seg = sq[0] == s_last;  // seq_idx is nondecreasing: no reset inside the chunk
      const bool tok_ok = i_row < len;
      const int si = tok_ok ? sq[i_row] : -2;
      const int lim = tok_ok ? i_row : -1;
      const bool fact = one_seg && f.A[ut[kUg] * hpg + hh] <= 0.0f;
      const float li = tok_ok ? lb[i_row] : lb[len - 1];
      const float r_row = wq > 0 ? __expf(li - lb[32 * wq]) : 0.0f;
      // this warp's factor table: exp(l_r - l_j) dt_j (l_r the l of the row
      // block's first row) for the columns of its units q = wg and wg + 4
      float* tab = wtab + warp * 32;
      if (fact && wg < 2 * wq) {  // warp-uniform: the warp has a factored unit
        const int j = lane < 16 ? 16 * wg + lane : 16 * (wg + 4) + lane - 16;
        tab[lane] = (j < 32 * wq && j < len) ? __expf(lb[32 * wq] - lb[j]) * db[j] : 0.0f;
        __syncwarp();
      }
      for (int q = wg; q <= 2 * wq + 1; q += 4) {
        const int j0 = q * 16;
        uint32_t pk[8] = {0, 0, 0, 0, 0, 0, 0, 0};
        if (j0 < len) {  // warp-uniform
          float v[16];
          tmem_ld16(tmem_addr(tCB, wlane, j0), v);
          if (fact && q < 2 * wq) {
            const float* s = tab + (q == wg ? 0 : 16);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const float4 sj = *reinterpret_cast<const float4*>(s + 4 * kk);
              pk[2 * kk] = pack2(v[4 * kk] * sj.x * r_row, v[4 * kk + 1] * sj.y * r_row);
              pk[2 * kk + 1] = pack2(v[4 * kk + 2] * sj.z * r_row, v[4 * kk + 3] * sj.w * r_row);
            }
          } else {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const float4 lj = *reinterpret_cast<const float4*>(lb + j0 + 4 * kk);
              const float4 dj = *reinterpret_cast<const float4*>(db + j0 + 4 * kk);
              int4 sj = make_int4(si, si, si, si);
              if (!one_seg) sj = *reinterpret_cast<const int4*>(sq + j0 + 4 * kk);
              const float lv[4] = {lj.x, lj.y, lj.z, lj.w}, dv[4] = {dj.x, dj.y, dj.z, dj.w};
              const int sv[4] = {sj.x, sj.y, sj.z, sj.w};
              float a[4];
#pragma unroll
              for (int m = 0; m < 4; ++m) {
                const bool on = j0 + 4 * kk + m <= lim && sv[m] == si;
                a[m] = v[4 * kk + m] * __expf(on ? li - lv[m] : -INFINITY) * dv[m];
              }
              pk[2 * kk] = pack2(a[0], a[1]);
              pk[2 * kk + 1] = pack2(a[2], a[3]);
            }
          }
        }
        uint8_t* blk = sA + (q >> 2) * kTok;
        const uint32_t e0 = (q & 3) * 16;
        *reinterpret_cast<uint4*>(blk + swz128_off(i_row, e0)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
        *reinterpret_cast<uint4*>(blk + swz128_off(i_row, e0 + 8)) = make_uint4(pk[4], pk[5], pk[6], pk[7]);
      }
      // this thread's scalar copies of head k+1 landed (visible to the other
      // warps after the next CTA-wide barrier, which precedes that head's passes)
      cp_async_wait_all();
      fence_async_smem();
      tc_fence_before();
      __syncwarp();  // the warp's part of M is written, its C B^T reads done
      if (lane == 0) mbar_arrive(b_mr);
    };

    // ---- epilogue of head e (head eh of unit eu): token t = r, headdim columns 16 wg ..
    auto epilogue = [&](int e, int eu, int eh) {
      const int us = eu % kRingU;
      const int* ut = utab + us * 8;
      const int* sq = sqr + us * kQ;
      const int slot = e % 3, buf = e & 1;
      const int h = ut[kUg] * hpg + eh, c = ut[kUc], t0 = ut[kUt0], len = ut[kUlen], bi = ut[kUbi];
      const long long bh = (long long)bi * p.H + h;
      const int s_last = sq[len - 1], s_in = ut[kUsin];
      const float* lb = lq + slot * kQ;
      const float* db = dtq + slot * kQ;
      const int t = r;
      const bool tv = t < len;
      const float Dh = __ldg(f.D + h);
      wait(b_b1, e & 1);
      wait(&b_xy[buf], (e >> 1) & 1);
      wait(&b_b2[buf], (e >> 1) & 1);
      tc_fence_after();
      const uint8_t* sX = sXb + buf * kTok;
      const uint8_t* sY = sYb + buf * kTok;
      const uint32_t tz = tZW + buf * 128, tw = tz + 64;
      // the accumulator rows in two halves (Z, dXs for dx; then W, Yc), so that
      // no more than 32 of them are live at once; the first half's reads are
      // in flight while the x, dy rows come from shared memory
      uint32_t zr[16], sr[16];
      tmem_ld16_issue(tmem_addr(tz, wlane, wg * 16), zr);
      tmem_ld16_issue(tmem_addr(tDXS, wlane, wg * 16), sr);
      uint4* y0p = reinterpret_cast<uint4*>(const_cast<uint8_t*>(sY) + swz128_off(t, wg * 16));
      uint4* y1p = reinterpret_cast<uint4*>(const_cast<uint8_t*>(sY) + swz128_off(t, wg * 16 + 8));
      const uint4 x0 = *reinterpret_cast<const uint4*>(sX + swz128_off(t, wg * 16));
      const uint4 x1 = *reinterpret_cast<const uint4*>(sX + swz128_off(t, wg * 16 + 8));
      const uint4 y0 = *y0p;
      const uint4 y1 = *y1p;
      tmem_ld_wait2(zr, sr);
      float z[16], s16[16];
#pragma unroll
      for (int kk = 0; kk < 16; ++kk) {
        z[kk] = __uint_as_float(zr[kk]);
        s16[kk] = __uint_as_float(sr[kk]);
      }
      const uint32_t xs[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
      const uint32_t ys[8] = {y0.x, y0.y, y0.z, y0.w, y1.x, y1.y, y1.z, y1.w};
      const float dtt = tv ? db[t] : 0.0f;
      const float lt = tv ? lb[t] : 0.0f;
      const float wt = (tv && sq[t] == s_last) ? __expf(lb[len - 1] - lt) : 0.0f;
      const float ut_ = wt * dtt;
      float zx = 0.0f, wy = 0.0f, du = 0.0f, ca = 0.0f, yx = 0.0f;
      uint32_t o[8];
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const float2 xv = unpack2(xs[kk]), yv = unpack2(ys[kk]);
        zx = fmaf(xv.x, z[2 * kk], fmaf(xv.y, z[2 * kk + 1], zx));
        du = fmaf(xv.x, s16[2 * kk], fmaf(xv.y, s16[2 * kk + 1], du));
        yx = fmaf(yv.x, xv.x, fmaf(yv.y, xv.y, yx));
        o[kk] = pack2(z[2 * kk] + fmaf(ut_, s16[2 * kk], Dh * yv.x),
                      z[2 * kk + 1] + fmaf(ut_, s16[2 * kk + 1], Dh * yv.y));
      }
      {
        float w16[16], y16[16];
        tmem_ld16x2(tmem_addr(tw, wlane, wg * 16), tmem_addr(tYC, wlane, wg * 16), w16, y16);
        // dXs and Yc of this head are read: the next head's may be formed
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(b_bf);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const float2 yv = unpack2(ys[kk]);
          wy = fmaf(yv.x, w16[2 * kk], fmaf(yv.y, w16[2 * kk + 1], wy));
          ca = fmaf(yv.x, y16[2 * kk], fmaf(yv.y, y16[2 * kk + 1], ca));
        }
      }
      // dx in place of this thread's dy row piece (already read), for the
      // tensor store of the whole tile (rows past the sequence are clipped)
      *y0p = make_uint4(o[0], o[1], o[2], o[3]);
      *y1p = make_uint4(o[4], o[5], o[6], o[7]);
      pZX[wg * kQ + t] = zx;
      pWY[wg * kQ + t] = wy;
      pDU[wg * kQ + t] = du;
      pCA[wg * kQ + t] = ca;
      pYX[wg * kQ + t] = tv ? yx : 0.0f;
      tc_fence_before();
      fence_async_smem();  // x and dy are next written by tensor copies (async proxy)
      named_sync_compute();  // TMEM pair, x, dy read back; partials complete
      if (tid == 0) mbar_arrive(&b_ed[e & 1]);
      if (wg == 0) {
        auto fold = [&](const float* a) { return (a[t] + a[kQ + t]) + (a[2 * kQ + t] + a[3 * kQ + t]); };
        const float colr = fold(pZX), roww = fold(pWY), dut = fold(pDU), car = fold(pCA);
        float udu = 0.0f;
        if (tv) {
          const float cv = sq[t] == s_in ? __expf(lt) : 0.0f;
          const float colq = dtt > 1e-30f ? colr / dtt : 0.0f;
          const float dd = colq + wt * dut;
          const float dl = roww - colr + cv * car - ut_ * dut;
          f.ddte[bh * p.Lp + t0 + t] = dd;
          f.dl[bh * p.Lp + t0 + t] = dl;
          udu = ut_ * dut;
        }
        // per-chunk sums: one slot per warp (row block), added in slot
        // order by the parameter-gradient kernels
        udu = warp_sum(udu);
        if (lane == 0) f.udu[(bh * p.nc + c) * p.cb_ntb + wq] = udu;
      } else if (wg == 1) {
        float v = (pYX[t] + pYX[kQ + t]) + (pYX[2 * kQ + t] + pYX[3 * kQ + t]);
        v = warp_sum(v);
        if (lane == 0) f.pdD[(((long long)bi * p.nc + c) * p.cb_ntb + wq) * p.H + h] = v;
      }
      // the partial arrays are next written after the next barrier, which
      // these readers pass only after reading them
    };

    // Per head k: the M tile of k, then the epilogue of k-1 while the tensor
    // core forms Z, W of k.  At the first head of a unit the epilogue of the
    // previous unit's last head goes first: it covers the copies of the new
    // unit's B, C and its C B^T.
    int iu = 0, hh = 0, eu = 0, eh = 0;  // unit and head of k, of k-1
    for (int k = 0; k <= nh; ++k) {
      const bool epi_first = k >= 1 && (k == nh || hh == 0);
      if (epi_first) epilogue(k - 1, eu, eh);
      if (k < nh) {
        mask_pass(k, iu, hh);
        if (k >= 1 && !epi_first) epilogue(k - 1, eu, eh);
        else named_sync_compute();  // the next head's scalars before its passes
      }
      eu = iu;
      eh = hh;
      if (++hh == hpg) {
        hh = 0;
        ++iu;
      }
    }
  }
  if (!ok) atomicOr(&f.hdr->status, kDevTimeout);
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tm, 512);
}

}  // namespace

bool chunk_bwd_tok_tc_supported(const Plan& p) {
  return p.dtype == SSD_BF16 && p.P == 64 && p.Q == kQ && (p.N == 16 || p.N == 32 || p.N == 64 || p.N == 128) &&
         p.hpg <= 256;
}

cudaError_t launch_chunk_bwd_tok_tc(const Plan& p, const Bufs& f, cudaStream_t s) {
  set_kernel_name("chunk_bwd_tc");
  const TokGeom T = tok_geom(p.N);
  CUtensorMap X, Y, B, C, S, H, DX;
  const uint64_t dbc[4] = {(uint64_t)p.N, (uint64_t)p.G, (uint64_t)p.L, (uint64_t)p.b};
  const uint64_t sbc[3] = {(uint64_t)p.N * 2, (uint64_t)p.G * p.N * 2, (uint64_t)p.L * p.G * p.N * 2};
  const uint32_t bbc[4] = {(uint32_t)(T.cw / 2), 1, (uint32_t)kQ, 1};
  const uint64_t dxx[4] = {64, (uint64_t)p.H, (uint64_t)p.L, (uint64_t)p.b};
  const uint64_t sxx[3] = {128, (uint64_t)p.H * 128, (uint64_t)p.L * p.H * 128};
  const uint32_t bxx[4] = {64, 1, (uint32_t)kQ, 1};
  const uint64_t ds[4] = {64, (uint64_t)p.N, (uint64_t)p.nc, (uint64_t)p.b * p.H};
  const uint64_t ss[3] = {128, (uint64_t)p.N * 128, (uint64_t)p.nc * p.N * 128};
  const uint32_t bs[4] = {64, (uint32_t)p.N, 1, 1};
  if (!encode_tmap_bf16_4d(&X, f.x, dxx, sxx, bxx, 128) || !encode_tmap_bf16_4d(&Y, f.dy, dxx, sxx, bxx, 128) ||
      !encode_tmap_bf16_4d(&B, f.B, dbc, sbc, bbc, T.cw) || !encode_tmap_bf16_4d(&C, f.C, dbc, sbc, bbc, T.cw) ||
      !encode_tmap_bf16_4d(&S, f.dS, ds, ss, bs, 128) || !encode_tmap_bf16_4d(&H, f.Hin, ds, ss, bs, 128) ||
      !encode_tmap_bf16_4d(&DX, f.dx, dxx, sxx, bxx, 128))
    return cudaErrorInvalidValue;
  const size_t smem = tok_smem_bytes(T);
  cudaError_t e = cudaFuncSetAttribute(chunk_bwd_tok_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  // one persistent CTA per SM (one fits: shared memory and all 512 TMEM
  // columns), at most one per work unit
  const long long units = (long long)p.nc * p.G * p.b;
  if (units >= (1ll << 31)) return cudaErrorInvalidValue;
  const long long sms = (p.flags & SSD_TEST_FEW_CTAS) ? 2 : device_sm_count();
  const int grid = (int)(units < sms ? units : sms);
  chunk_bwd_tok_tc_kernel<<<grid, kThr, smem, s>>>(p, f, X, Y, B, C, S, H, DX);
  return cudaGetLastError();
}

}  // namespace ssd
