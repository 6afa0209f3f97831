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
// One CTA per (chunk, group, batch row): 16 compute warps (warp w reads TMEM
// lane quarter w % 4) and two control warps, one lane of each issuing.
//   control A: the tile copies, C B^T once, per head dXs = B dS^T, Yc = C H^T;
//   control B: per head Z = M^T dY and W = M X into a double-buffered pair;
//   compute, per head hh: the M tile (units strictly below a row block's
//     diagonal block use exp(l_i - l_r) exp(l_r - l_j) dt_j, l_r the block's
//     first row, both exponentials <= 1, the second from a per-head table),
//     then the epilogue of head hh-1 while the tensor core forms Z, W of
//     head hh.
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

// floats after offF: l, dt [3 slots][Q]; segment ids [Q]; factor table
// [3][Q]; five partial arrays [4][Q]; per-warp sums [8]; then the barriers,
// the TMEM address and D of the group's heads
constexpr int kFloats = 3 * kQ + 3 * kQ + kQ + 3 * kQ + 20 * kQ + 8;

__host__ __device__ inline size_t tok_smem_bytes(const TokGeom& T, int hpg) {
  return 1024 + T.offF + (size_t)kFloats * 4 + 16 * 8 + 16 + (size_t)hpg * 4 + 16;
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
  int* sq = reinterpret_cast<int*>(dtq + 3 * kQ);     // [Q]
  float* sfac = reinterpret_cast<float*>(sq + kQ);    // [3][Q] exp(l_{32 rb} - l_j) dt_j, rb = 1..3
  float* pZX = sfac + 3 * kQ;                         // [4 warpgroups][Q] x . Z
  float* pWY = pZX + 4 * kQ;                          // dy . W
  float* pDU = pWY + 4 * kQ;                          // x . dXs
  float* pCA = pDU + 4 * kQ;                          // dy . Yc
  float* pYX = pCA + 4 * kQ;                          // dy . x
  float* red = pYX + 4 * kQ;                          // [8]
  uint64_t* bar = reinterpret_cast<uint64_t*>(red + 8);
  uint64_t *b_bc = bar, *b_xy = bar + 1, *b_sh = bar + 3, *b_cb = bar + 4, *b_b1 = bar + 5, *b_mr = bar + 6,
           *b_b2 = bar + 7, *b_ed = bar + 9;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + 16);
  float* sD = reinterpret_cast<float*>(tmem_slot + 4);  // [hpg]

  const int c = blockIdx.x, g = blockIdx.y, bi = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int wg = (tid >> 7) & 3, r = tid & 127, wq = (tid >> 5) & 3;
  const int wlane = wq * 32;
  const int t0 = c * kQ, len = min(kQ, p.L - t0);
  const int hpg = p.hpg, h_first = g * hpg;
  const long long bh0 = (long long)bi * p.H + h_first;
  const uint32_t c_bytes = (uint32_t)T.ncb * T.cblk;
  const uint32_t s_bytes = (uint32_t)p.N * 128u;
  auto issue_xy = [&](int hh) {
    const int buf = hh & 1, h = h_first + hh;
    mbar_expect_tx(&b_xy[buf], 2 * kTok);
    tma_load_4d(sXb + buf * kTok, &tmX, &b_xy[buf], 0, h, t0, bi);
    tma_load_4d(sYb + buf * kTok, &tmY, &b_xy[buf], 0, h, t0, bi);
  };
  auto issue_sh = [&](int hh) {
    const int h = h_first + hh;
    mbar_expect_tx(b_sh, 2 * s_bytes);
    tma_load_4d(sS, &tmS, b_sh, 0, 0, c, bi * p.H + h);
    tma_load_4d(sH, &tmH, b_sh, 0, 0, c, bi * p.H + h);
  };
  if (tid == kCompute) {  // control A starts the tile copies first
    for (int k = 0; k < 10; ++k) mbar_init(&bar[k], 1);  // bc, xy[2], sh, cb, b1, mr, b2[2], ed
    mbar_fence_init();
    mbar_expect_tx(b_bc, 2 * c_bytes);
    for (int q = 0; q < T.ncb; ++q) {
      tma_load_4d(sB + q * T.cblk, &tmB, b_bc, q * 64, g, t0, bi);
      tma_load_4d(sC + q * T.cblk, &tmC, b_bc, q * 64, g, t0, bi);
    }
    issue_xy(0);
    if (hpg > 1) issue_xy(1);
    issue_sh(0);
  }
  for (int t = tid; t < kQ; t += kThr) sq[t] = t < len ? seg_of(p, f, bi, (long long)t0 + t) : -1;
  if (tid < kQ) {  // scalars of the group's first head into slot 0
    lq[tid] = f.lcs[bh0 * p.Lp + t0 + tid];
    dtq[tid] = f.dte[bh0 * p.Lp + t0 + tid];
  }
  for (int k = tid; k < hpg; k += kThr) sD[k] = f.D[h_first + k];
  if (warp == 0) tmem_alloc(tmem_slot, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tm = *tmem_slot;
  // C B^T | [2] (Z | W) | dXs | Yc
  const uint32_t tCB = tm, tZW = tm + 128, tDXS = tm + 384, tYC = tm + 448;
  bool ok = true;
  auto wait = [&](uint64_t* b, uint32_t ph) {
    if (!mbar_wait(b, ph)) ok = false;
  };

  if (warp >= kCompute / 32) {
    const int cw = warp - kCompute / 32;
    if (lane == 0) {
      const uint32_t id128 = idesc_bf16(128, 128, 0, 0), id64 = idesc_bf16(128, 64, 0, 1);
      const uint32_t id64t = idesc_bf16(128, 64, 1, 1);
      auto kdesc_c = [&](const uint8_t* t, int ks) {  // K-major B/C tile, K = d_state
        const uint32_t kb = (ks * 32) / T.cw, kin = (ks * 32) % T.cw;
        return smem_desc(smem_u32(t) + kb * T.cblk + kin, 16, 8 * T.cw, T.cswz);
      };
      auto mndesc_rows = [&](const uint8_t* t, int ks) {  // MN-major (64 wide), K along rows
        return smem_desc(smem_u32(t) + ks * 16 * 128, 16, 1024, kSwz128);
      };
      if (cw == 0) {
        // ---------------- control A: copies, C B^T, per head dXs and Yc ----------------
        wait(b_bc, 0);
        tc_fence_after();
        for (int ks = 0; ks < p.N / 16; ++ks)  // C B^T (M = i, N = j, K = d_state), once per group
          mma_bf16(tCB, kdesc_c(sC, ks), kdesc_c(sB, ks), id128, ks > 0);
        mma_commit(b_cb);
        for (int hh = 0; hh < hpg; ++hh) {
          wait(b_sh, hh & 1);
          if (hh >= 1) {
            // the epilogue of head hh-1 has read dXs, Yc and its x, dy buffer
            // and left that head's dx in the dy tile: store it, then refill
            // the buffer once the store has read it
            wait(b_ed, (hh - 1) & 1);
            tma_store_4d(&tmDX, sYb + ((hh - 1) & 1) * kTok, 0, h_first + hh - 1, t0, bi);
            bulk_commit();
            if (hh + 1 < hpg) {
              bulk_wait_read<0>();
              issue_xy(hh + 1);
            }
          }
          tc_fence_after();
          for (int ks = 0; ks < p.N / 16; ++ks) {
            mma_bf16(tDXS, kdesc_c(sB, ks), mndesc_rows(sS, ks), id64, ks > 0);
            mma_bf16(tYC, kdesc_c(sC, ks), mndesc_rows(sH, ks), id64, ks > 0);
          }
          mma_commit(b_b1);
          if (hh + 1 < hpg) {
            wait(b_b1, hh & 1);  // dS, H read
            issue_sh(hh + 1);
          }
        }
        wait(b_ed, (hpg - 1) & 1);  // the last head's dx
        tma_store_4d(&tmDX, sYb + ((hpg - 1) & 1) * kTok, 0, h_first + hpg - 1, t0, bi);
        bulk_commit();
        bulk_wait_all();
      } else {
        // ---------------- control B: per head Z = M^T dY, W = M X ----------------
        for (int hh = 0; hh < hpg; ++hh) {
          // M of head hh written; the pair hh & 1 was read by the epilogue
          // of head hh-2, which the compute warps finished first; x, dy of
          // head hh landed (the mask pass does not read them)
          wait(b_mr, hh & 1);
          wait(&b_xy[hh & 1], (hh >> 1) & 1);
          tc_fence_after();
          const uint32_t tz = tZW + (hh & 1) * 128, tw = tz + 64;
          const uint8_t* sY = sYb + (hh & 1) * kTok;
          const uint8_t* sX = sXb + (hh & 1) * kTok;
          for (int ks = 0; ks < kQ / 16; ++ks) {
            const uint64_t am = smem_desc(smem_u32(sA) + ks * 16 * 128, kTok, 1024, kSwz128);   // M^T
            const uint64_t ak = smem_desc(smem_u32(sA) + (ks / 4) * kTok + (ks % 4) * 32, 16, 1024, kSwz128);
            mma_bf16(tz, am, mndesc_rows(sY, ks), id64t, ks > 0);
            mma_bf16(tw, ak, mndesc_rows(sX, ks), id64, ks > 0);
          }
          mma_commit(&b_b2[hh & 1]);
        }
      }
    }
  } else {
    // ---------------- 16 compute warps ----------------
    const int s_in = seg_in_of(p, f, bi, c);
    const int s_last = sq[len - 1];
    const bool one_seg = sq[0] == s_last;  // seq_idx is nondecreasing: no reset inside the chunk
    const int i = wlane + lane;            // row of this thread in the mask pass
    const bool tok_ok = i < len;
    const int si = tok_ok ? sq[i] : -2;
    const int lim = tok_ok ? i : -1;
    // per-head factor table exp(l_{32 rb} - l_j) (j < 32 rb), from slot `slot`
    auto fill_fac = [&](int slot) {
      if (tid < 3 * kQ) {
        const int rb = 1 + tid / kQ, j = tid % kQ;
        const float* lb = lq + slot * kQ;
        const float* db = dtq + slot * kQ;
        sfac[tid] = (j < 32 * rb && j < len) ? __expf(lb[32 * rb] - lb[j]) * db[j] : 0.0f;
      }
    };
    fill_fac(0);
    // upper-triangle 16-column units of the M tile: zero once
    for (int q = 2 * wq + 2 + wg; q < 8; q += 4) {
      uint8_t* blk = sA + (q >> 2) * kTok;
      const uint32_t e0 = (q & 3) * 16;
      *reinterpret_cast<uint4*>(blk + swz128_off(i, e0)) = make_uint4(0, 0, 0, 0);
      *reinterpret_cast<uint4*>(blk + swz128_off(i, e0 + 8)) = make_uint4(0, 0, 0, 0);
    }
    named_sync_compute();
    wait(b_cb, 0);
    tc_fence_after();
    for (int hh = 0; hh <= hpg; ++hh) {
      if (hh < hpg) {
        const int slot = hh % 3;
        const float* lb = lq + slot * kQ;
        const float* db = dtq + slot * kQ;
        if (hh + 1 < hpg && tid < kQ) {  // scalars of head hh+1 (slot last read by head hh-2)
          const int sn = (hh + 1) % 3;
          cp_async4(lq + sn * kQ + tid, f.lcs + (bh0 + hh + 1) * p.Lp + t0 + tid);
          cp_async4(dtq + sn * kQ + tid, f.dte + (bh0 + hh + 1) * p.Lp + t0 + tid);
        }
        cp_async_commit();
        if (hh >= 1) {  // Z, W of head hh-1 done: M may be rewritten
          wait(&b_b2[(hh - 1) & 1], ((hh - 1) >> 1) & 1);
          tc_fence_after();
        }
        // ---- M tile: row i, 16-column units of this row block
        const bool fact = one_seg && f.A[h_first + hh] <= 0.0f;
        const float li = tok_ok ? lb[i] : lb[len - 1];
        const float r_row = wq > 0 ? __expf(li - lb[32 * wq]) : 0.0f;
        for (int q = wg; q <= 2 * wq + 1; q += 4) {
          const int j0 = q * 16;
          uint32_t pk[8] = {0, 0, 0, 0, 0, 0, 0, 0};
          if (j0 < len) {  // warp-uniform
            float v[16];
            tmem_ld16(tmem_addr(tCB, wlane, j0), v);
            if (fact && q < 2 * wq) {
              const float* s = sfac + (wq - 1) * kQ;
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                const float4 sj = *reinterpret_cast<const float4*>(s + j0 + 4 * k);
                pk[2 * k] = pack2(v[4 * k] * sj.x * r_row, v[4 * k + 1] * sj.y * r_row);
                pk[2 * k + 1] = pack2(v[4 * k + 2] * sj.z * r_row, v[4 * k + 3] * sj.w * r_row);
              }
            } else {
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                const float4 lj = *reinterpret_cast<const float4*>(lb + j0 + 4 * k);
                const float4 dj = *reinterpret_cast<const float4*>(db + j0 + 4 * k);
                int4 sj = make_int4(si, si, si, si);
                if (!one_seg) sj = *reinterpret_cast<const int4*>(sq + j0 + 4 * k);
                const float lv[4] = {lj.x, lj.y, lj.z, lj.w}, dv[4] = {dj.x, dj.y, dj.z, dj.w};
                const int sv[4] = {sj.x, sj.y, sj.z, sj.w};
                float a[4];
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                  const bool on = j0 + 4 * k + m <= lim && sv[m] == si;
                  a[m] = v[4 * k + m] * __expf(on ? li - lv[m] : -INFINITY) * dv[m];
                }
                pk[2 * k] = pack2(a[0], a[1]);
                pk[2 * k + 1] = pack2(a[2], a[3]);
              }
            }
          }
          uint8_t* blk = sA + (q >> 2) * kTok;
          const uint32_t e0 = (q & 3) * 16;
          *reinterpret_cast<uint4*>(blk + swz128_off(i, e0)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
          *reinterpret_cast<uint4*>(blk + swz128_off(i, e0 + 8)) = make_uint4(pk[4], pk[5], pk[6], pk[7]);
        }
        cp_async_wait_all();  // scalars of head hh+1 landed (visible after the barrier)
        fence_async_smem();
        tc_fence_before();
        named_sync_compute();  // M complete; C B^T reads of this head done
        if (tid == 0) mbar_arrive(b_mr);
        // factor table of the next head: its scalars are visible since the
        // barrier, and this head's mask pass is done with the table; the
        // epilogue's barriers (or the one below) order it before that head's
        // mask pass
        if (hh + 1 < hpg) fill_fac((hh + 1) % 3);
        if (hh == 0) named_sync_compute();
      }
      if (hh >= 1) {
        // ---- epilogue of head e = hh - 1: token t = r, headdim columns 16 wg ..
        const int e = hh - 1, slot = e % 3, buf = e & 1, h = h_first + e;
        const long long bh = bh0 + e;
        const float* lb = lq + slot * kQ;
        const float* db = dtq + slot * kQ;
        const int t = r;
        const bool tv = t < len;
        wait(b_b1, e & 1);
        wait(&b_xy[buf], (e >> 1) & 1);
        if (hh == hpg) wait(&b_b2[buf], (e >> 1) & 1);
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
        for (int k = 0; k < 16; ++k) {
          z[k] = __uint_as_float(zr[k]);
          s16[k] = __uint_as_float(sr[k]);
        }
        const uint32_t xs[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
        const uint32_t ys[8] = {y0.x, y0.y, y0.z, y0.w, y1.x, y1.y, y1.z, y1.w};
        const float dtt = tv ? db[t] : 0.0f;
        const float lt = tv ? lb[t] : 0.0f;
        const float wt = (tv && sq[t] == s_last) ? __expf(lb[len - 1] - lt) : 0.0f;
        const float ut = wt * dtt;
        const float Dh = sD[e];
        float zx = 0.0f, wy = 0.0f, du = 0.0f, ca = 0.0f, yx = 0.0f;
        uint32_t o[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const float2 xv = unpack2(xs[k]), yv = unpack2(ys[k]);
          zx = fmaf(xv.x, z[2 * k], fmaf(xv.y, z[2 * k + 1], zx));
          du = fmaf(xv.x, s16[2 * k], fmaf(xv.y, s16[2 * k + 1], du));
          yx = fmaf(yv.x, xv.x, fmaf(yv.y, xv.y, yx));
          o[k] = pack2(z[2 * k] + fmaf(ut, s16[2 * k], Dh * yv.x),
                       z[2 * k + 1] + fmaf(ut, s16[2 * k + 1], Dh * yv.y));
        }
        {
          float w16[16], y16[16];
          tmem_ld16x2(tmem_addr(tw, wlane, wg * 16), tmem_addr(tYC, wlane, wg * 16), w16, y16);
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const float2 yv = unpack2(ys[k]);
            wy = fmaf(yv.x, w16[2 * k], fmaf(yv.y, w16[2 * k + 1], wy));
            ca = fmaf(yv.x, y16[2 * k], fmaf(yv.y, y16[2 * k + 1], ca));
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
        named_sync_compute();  // TMEM pair, dXs, Yc, x, dy read back; partials complete
        if (tid == 0) mbar_arrive(b_ed);
        if (wg == 0) {
          auto fold = [&](const float* a) { return (a[t] + a[kQ + t]) + (a[2 * kQ + t] + a[3 * kQ + t]); };
          const float colr = fold(pZX), roww = fold(pWY), dut = fold(pDU), car = fold(pCA);
          float udu = 0.0f;
          if (tv) {
            const float cv = sq[t] == s_in ? __expf(lt) : 0.0f;
            const float colq = dtt > 1e-30f ? colr / dtt : 0.0f;
            const float dd = colq + wt * dut;
            const float dl = roww - colr + cv * car - ut * dut;
            f.ddte[bh * p.Lp + t0 + t] = dd;
            f.dl[bh * p.Lp + t0 + t] = dl;
            udu = ut * dut;
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
  const size_t smem = tok_smem_bytes(T, p.hpg);
  cudaError_t e = cudaFuncSetAttribute(chunk_bwd_tok_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  chunk_bwd_tok_tc_kernel<<<dim3(p.nc, p.G, p.b), kThr, smem, s>>>(p, f, X, Y, B, C, S, H, DX);
  return cudaGetLastError();
}

}  // namespace ssd
