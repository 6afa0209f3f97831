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
// streamed.  Warp-specialised: one control warp issues every TMA copy (x and
// carry-in-state tiles of the next head into a double buffer) and every MMA;
// sixteen compute warps (four per quarter of the TMEM lanes, one lane = one
// row) read C B^T back, apply the causal / same-sequence mask,
// exp(l_i - l_j) and dt_eff_j of the head, write the bf16 K-major A_hat tile
// (two A_hat buffers where shared memory allows, chunk <= 128), then run the
// epilogue y = Y1 + cv e^{l} Y2 + D x of the previous head while the tensor
// core computes Y1 = A_hat X and the carry Y2 = C H_in^T of this one into a
// double-buffered accumulator pair.  The two sides meet only at mbarriers
// (A_hat written, MMAs done, accumulators read back), so no block-wide
// barrier waits on the thread that issues the MMAs.  Per-head l and dt_eff
// are prefetched two heads ahead into a ring of three shared-memory slots,
// the epilogue's x row one head ahead into registers.  With chunk = 128 the
// mask work is balanced over the lane quarters (see the mask pass).
#include "ssd_internal.cuh"
#include "tc_common.cuh"
#include "tma_host.h"

namespace ssd {

namespace {

using namespace tc;

constexpr int kRows = 128;  // rows (tokens i) per CTA = MMA M
constexpr int kCompute = 512;         // 16 compute warps: four per quarter of the TMEM lanes
constexpr int kThr = kCompute + 32;   // and one control warp that issues the copies and MMAs

__host__ __device__ inline uint32_t r1024(uint32_t v) { return (v + 1023u) & ~1023u; }

struct ScanGeom {
  int rows;          // tokens per TMA box = min(Q, 128)
  int nJ;            // column blocks (== number of row blocks)
  int cw, ncb;       // bytes per row of one B/C column block, column blocks along d_state
  uint32_t cblk;     // bytes of one B/C column block (kRows rows)
  uint32_t cswz;     // swizzle code of B/C tiles
  uint32_t cbytes;   // bytes of one B or C tile
  uint32_t offC, offB, offX, offH, offA2, offCr, offYs, offF, bytes;
  int nys;           // y staging buffers (each: 16 warps x 32 rows x 32 bytes)
  bool dbl;          // a second A_hat buffer fits: the mask pass of head h+1 overlaps the MMAs of head h
  bool bal;          // chunk = 128: the causal mask work is balanced over the four lane quarters
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
  g.offA2 = g.offH + 2u * r1024((uint32_t)N * 128u);
  const uint32_t ys = (uint32_t)kCompute * 32u;  // one y staging buffer
  const uint32_t lim = 227u * 1024u - (1024u + 8u * 256u * 4u + 512u);  // minus alignment and scalars
  g.dbl = g.offA2 + g.nJ * bsp + ys <= lim;
  g.offCr = g.offA2 + (g.dbl ? g.nJ * bsp : 0u);
  // C_rev is only read by the MMA that forms C_rev B^T; after it, its space
  // can hold the y staging buffers when it is large enough
  const bool ys_in_cr = g.cbytes >= 2u * ys;
  g.bal = Q == kRows && g.dbl && g.offCr + g.cbytes + (ys_in_cr ? 0u : ys) <= lim;
  if (g.bal && ys_in_cr) {
    g.offYs = g.offCr;
    g.nys = 2;
    g.offF = g.offCr + g.cbytes;
  } else {
    g.offYs = g.offCr + (g.bal ? g.cbytes : 0u);
    g.nys = g.offYs + 2u * ys <= lim ? 2 : 1;
    g.offF = g.offYs + g.nys * ys;
  }
  g.bytes = g.offF;
  return g;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

// One warp-uniform unit of the mask pass: this thread's row `tok`
// (chunk-local) against the 16 columns j0 .. j0+15.  A_hat entry =
// (C_tok . B_j) exp(l_tok - l_j) dt_j for j <= tok in the same segment, else
// 0 (exp of -inf).  Branch-free: the column scalars come as float4
// broadcasts from shared memory.
__device__ __forceinline__ void mask_unit(const float (&v)[16], const float* l2, const float* dtv, const int* sq,
                                          int j0, int lim, int st, float lt2, bool one_seg, uint32_t (&pk)[8]) {
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float4 lj = *reinterpret_cast<const float4*>(l2 + j0 + 4 * k);
    const float4 dj = *reinterpret_cast<const float4*>(dtv + j0 + 4 * k);
    int4 sj = make_int4(st, st, st, st);
    if (!one_seg) sj = *reinterpret_cast<const int4*>(sq + j0 + 4 * k);
    const float lv[4] = {lj.x, lj.y, lj.z, lj.w}, dv[4] = {dj.x, dj.y, dj.z, dj.w};
    const int sv[4] = {sj.x, sj.y, sj.z, sj.w};
    float a[4];
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      const bool on = j0 + 4 * k + m <= lim && sv[m] == st;
      a[m] = v[4 * k + m] * __expf(on ? lt2 - lv[m] : -INFINITY) * dv[m];
    }
    pk[2 * k] = pack_bf16x2(a[0], a[1]);
    pk[2 * k + 1] = pack_bf16x2(a[2], a[3]);
  }
}

__device__ __forceinline__ void named_sync_compute() {  // the 16 compute warps only
  asm volatile("bar.sync 1, %0;" ::"n"(kCompute) : "memory");
}

__global__ void __launch_bounds__(kThr, 1) chunk_scan_tc_kernel(Plan p, Bufs f,
                                                                const __grid_constant__ CUtensorMap tmC,
                                                                const __grid_constant__ CUtensorMap tmB,
                                                                const __grid_constant__ CUtensorMap tmX,
                                                                const __grid_constant__ CUtensorMap tmH,
                                                                const __grid_constant__ CUtensorMap tmC32,
                                                                const __grid_constant__ CUtensorMap tmY) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const ScanGeom G = scan_geom(p.N, p.Q);
  const uint32_t abytes = 2u * kRows * 128u;
  const uint32_t bsp = G.cbytes > abytes ? G.cbytes : abytes;
  const int I = blockIdx.x % G.nJ, c = blockIdx.x / G.nJ;
  const int g = blockIdx.y, bi = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31;
  const bool ctl = tid >= kCompute;  // the control warp: TMA and MMA issue
  const int wg = (tid >> 7) & 3;     // compute warpgroup: column quarter of the mask pass
  const int ri = tid & 127;          // row (TMEM lane) of this compute thread
  const int wlane = ((tid >> 5) & 3) * 32;
  const int t0 = c * p.Q, len = min(p.Q, p.L - t0);
  const int i0 = I * kRows;
  if (i0 >= len) return;  // row block past the ragged end (uniform per CTA)
  const int nJ = I + 1;   // column blocks J <= I
  uint8_t* sC = sm + G.offC;
  uint8_t* sB = sm + G.offB;  // B_J tiles, then A_hat_J tiles
  uint8_t* sX = sm + G.offX;
  uint8_t* sH = sm + G.offH;
  uint8_t* sA2 = sm + G.offA2;  // second A_hat buffer (when G.dbl)
  uint8_t* sCr = sm + G.offCr;  // C with its four 32-row blocks in reverse order (when G.bal)
  uint8_t* sYs = sm + G.offYs;  // [nys][16 warps][32 rows][32 B]: y staging for the tensor stores
  const uint32_t hbytes = r1024((uint32_t)p.N * 128u);
  float* lq = reinterpret_cast<float*>(sm + G.offF);   // [3][Q] l of a head, ring of 3 heads
  float* dq = lq + 3 * p.Q;                            // [3][Q]
  int* sq = reinterpret_cast<int*>(dq + 3 * p.Q);      // [Q]
  // xh[2] (TMA x, H_in), ld (C, B), cb (C B^T formed), ahat[2] (A_hat written),
  // mmad[2] (head MMAs done), yfree[2] (accumulator pair read back)
  uint64_t* bar = reinterpret_cast<uint64_t*>(sq + p.Q);
  uint64_t *b_xh = bar, *b_ld = bar + 2, *b_cb = bar + 3, *b_ahat = bar + 4, *b_mmad = bar + 6,
           *b_yfree = bar + 8;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + 10);
  float* sD = reinterpret_cast<float*>(tmem_slot + 4);  // [hpg] D of the group's heads
  const int hpg = p.hpg, h_first = g * hpg;
  const uint32_t xbox = (uint32_t)G.rows * 128u;
  auto issue_head = [&](int hh) {  // x tiles (J <= I) and carry-in state of head hh -> buffer hh&1
    const int buf = hh & 1, h = h_first + hh;
    mbar_expect_tx(&b_xh[buf], nJ * xbox + (uint32_t)p.N * 128u);
    for (int J = 0; J < nJ; ++J)
      tma_load_4d(sX + (buf * G.nJ + J) * kRows * 128, &tmX, &b_xh[buf], 0, h, t0 + J * kRows, bi);
    tma_load_4d(sH + buf * hbytes, &tmH, &b_xh[buf], 0, 0, c, bi * p.H + h);
  };
  if (tid == kCompute) {  // the control lane starts the tile copies before anything else
    const uint32_t cbox = (uint32_t)G.rows * G.cw;
    mbar_init(b_ld, 1);
    mbar_init(&b_xh[0], 1);
    mbar_init(&b_xh[1], 1);
    mbar_fence_init();
    // C_I and every B_J (J <= I) for C B^T; C_rev for C_rev B^T
    mbar_expect_tx(b_ld, (1 + nJ + (G.bal ? 1 : 0)) * G.ncb * cbox);
    for (int q = 0; q < G.ncb; ++q) {
      tma_load_4d(sC + q * G.cblk, &tmC, b_ld, q * 64, g, t0 + i0, bi);
      for (int J = 0; J < nJ; ++J)
        tma_load_4d(sB + J * bsp + q * G.cblk, &tmB, b_ld, q * 64, g, t0 + J * kRows, bi);
      if (G.bal)  // row block rb of C_rev is row block 3 - rb of C
        for (int rb = 0; rb < 4; ++rb)
          tma_load_4d(sCr + q * G.cblk + rb * 32 * G.cw, &tmC32, b_ld, q * 64, g, t0 + 32 * (3 - rb), bi);
    }
    issue_head(0);
    if (hpg > 1) issue_head(1);
  }
  for (int k = tid; k < hpg; k += kThr) sD[k] = f.D[h_first + k];

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
    for (int k = 3; k < 8; ++k) mbar_init(&bar[k], 1);
    mbar_init(&b_yfree[0], kCompute / 32);  // one arrival per compute warp
    mbar_init(&b_yfree[1], kCompute / 32);
    mbar_fence_init();
  }
  if (tid < 32) tmem_alloc(tmem_slot, 512);
  fence_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tm = *tmem_slot;
  const uint32_t tCB = tm;                 // nJ x 128 columns
  const uint32_t tCB2 = tm + 128;          // (G.bal) C_rev B^T: lane quarter s holds rows of block 3-s
  const uint32_t tY = tm + 256;            // [2 buffers] x (Y1 64 | Y2 64)
  bool ok = true;

  if (ctl) {
    // ---------------- control warp: one lane issues every copy and MMA ----------------
    if (lane == 0) {
      auto mma_ck = [&](uint32_t d, const uint8_t* a, const uint8_t* b, int kdim, uint32_t idesc, bool b_mn) {
        for (int ks = 0; ks < kdim / 16; ++ks) {
          const uint32_t kb = (ks * 32) / G.cw, kin = (ks * 32) % G.cw;
          const uint64_t da = smem_desc(smem_u32(a) + kb * G.cblk + kin, 16, 8 * G.cw, G.cswz);
          const uint64_t db = b_mn ? smem_desc(smem_u32(b) + ks * 16 * 128, 16, 1024, kSwz128)
                                   : smem_desc(smem_u32(b) + kb * G.cblk + kin, 16, 8 * G.cw, G.cswz);
          mma_bf16(d, da, db, idesc, ks > 0 ? 1u : 0u);
        }
      };
      if (!mbar_wait(b_ld, 0)) ok = false;
      tc_fence_after();
      for (int J = 0; J < nJ; ++J)
        mma_ck(tCB + J * 128, sC, sB + J * bsp, p.N, idesc_bf16(128, 128, 0, 0), false);
      if (G.bal) mma_ck(tCB2, sCr, sB, p.N, idesc_bf16(128, 128, 0, 0), false);
      mma_commit(b_cb);
      const uint32_t id64 = idesc_bf16(128, 64, 0, 1);
      for (int hh = 0; hh < hpg; ++hh) {
        const int buf = hh & 1;
        if (!mbar_wait(&b_ahat[buf], (hh >> 1) & 1)) ok = false;                // A_hat of head hh
        if (hh >= 2 && !mbar_wait(&b_yfree[buf], ((hh - 2) >> 1) & 1)) ok = false;  // Y pair read
        if (!mbar_wait(&b_xh[buf], (hh >> 1) & 1)) ok = false;                  // x, H_in of head hh
        tc_fence_after();
        const uint8_t* sA = (G.dbl && buf) ? sA2 : sB;
        const uint32_t d1 = tY + buf * 128, d2 = d1 + 64;
        const uint8_t* xb = sX + buf * G.nJ * kRows * 128;
        for (int J = 0; J < nJ; ++J)
          for (int ks = 0; ks < kRows / 16; ++ks) {  // Y1 += A_hat_J X_J
            const uint64_t da =
                smem_desc(smem_u32(sA + J * bsp) + (ks / 4) * (kRows * 128) + (ks % 4) * 32, 16, 1024, kSwz128);
            const uint64_t dbx = smem_desc(smem_u32(xb + J * kRows * 128) + ks * 16 * 128, 16, 1024, kSwz128);
            mma_bf16(d1, da, dbx, id64, (J > 0 || ks > 0) ? 1u : 0u);
          }
        mma_ck(d2, sC, sH + buf * hbytes, p.N, id64, true);  // Y2 = C_I H^T
        mma_commit(&b_mmad[buf]);
        if (hh >= 1 && hh + 1 < hpg) {  // head hh+1 into the x/state buffer that head hh-1 used,
          // once the epilogue of head hh-1 has read its x rows (it waited for its MMAs first)
          if (!mbar_wait(&b_yfree[buf ^ 1], ((hh - 1) >> 1) & 1)) ok = false;
          issue_head(hh + 1);
        }
      }
    }
  } else {
    // ---------------- 16 compute warps: mask pass and epilogue ----------------
    const int i = i0 + ri;
    const bool row_ok = i < len;
    const int si = row_ok ? sq[i] : -2;
    const int s_in = seg_in_of(p, f, bi, c);
    const bool one_seg = sq[0] == sq[len - 1];  // seq_idx is nondecreasing: no reset inside the chunk
    // y rows of head hh: Y1 + cv e^{l} Y2 + D x from accumulator pair hh&1 and
    // the head's x tile (still resident: the control warp refills it only
    // after this epilogue released it); staged per warp (32 rows x 16
    // columns) and written by a tensor store.  li (the row's l of head hh) and
    // Dh were read before the ring slot could be refilled.
    const int warp = tid >> 5;
    auto epilogue = [&](int hh, float li, float Dh) {
      const int buf = hh & 1, h = h_first + hh;
      if (!mbar_wait(&b_mmad[buf], (hh >> 1) & 1)) ok = false;
      tc_fence_after();
      const float carry = (row_ok && si == s_in) ? __expf(li) : 0.0f;
      const int q = wg;  // the four warpgroups split the 64 output columns
      const uint8_t* xt = sX + (buf * G.nJ + I) * kRows * 128;
      const uint4 x0 = *reinterpret_cast<const uint4*>(xt + swz128_off(ri, q * 16));
      const uint4 x1 = *reinterpret_cast<const uint4*>(xt + swz128_off(ri, q * 16 + 8));
      float a[16], b[16];
      tmem_ld16x2(tmem_addr(tY + buf * 128, wlane, q * 16), tmem_addr(tY + buf * 128 + 64, wlane, q * 16), a, b);
      tc_fence_before();
      fence_async_smem();  // the x tile is next written by a tensor copy (async proxy)
      __syncwarp();
      if (lane == 0) mbar_arrive(&b_yfree[buf]);  // accumulator pair and x tile released
      const uint32_t xs[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
      uint32_t o[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float2 xf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&xs[e]));
        o[e] = pack_bf16x2(a[2 * e] + carry * b[2 * e] + Dh * xf.x, a[2 * e + 1] + carry * b[2 * e + 1] + Dh * xf.y);
      }
      uint8_t* yst = sYs + ((hh % G.nys) * (kCompute / 32) + warp) * 1024;
      if (lane == 0 && hh >= G.nys) {  // the store that last read this staging block has read it
        if (G.nys == 2) bulk_wait_read<1>();
        else bulk_wait_read<0>();
      }
      __syncwarp();
      *reinterpret_cast<uint4*>(yst + lane * 32) = make_uint4(o[0], o[1], o[2], o[3]);
      *reinterpret_cast<uint4*>(yst + lane * 32 + 16) = make_uint4(o[4], o[5], o[6], o[7]);
      fence_async_smem();
      __syncwarp();
      // rows past the end of the sequence are outside the tensor and not
      // written; rows past a short chunk (chunk 64) belong to the next chunk
      if (lane == 0 && i0 + wlane < G.rows * G.nJ) {
        tma_store_4d(&tmY, yst, q * 16, h, t0 + i0 + wlane, bi);
        bulk_commit();
      }
    };

    if (!mbar_wait(b_cb, 0)) ok = false;  // C B^T (and C_rev B^T) in tensor memory
    tc_fence_after();
    float li_prev = 0.0f, d_prev = 0.0f;
    for (int hh = 0; hh < hpg; ++hh) {
      const int buf = hh & 1;
      // asynchronous prefetch, for later in this iteration: the x row of head
      // hh-1 (epilogue) and the scalars of head hh+2 into ring slot (hh+2)%3,
      // whose last readers (the mask pass of head hh-1 and the l of its rows)
      // finished before the previous barrier
      const int pre = hh + 2;
      if (pre < hpg && tid < p.Q) {  // Q <= 256 < kCompute: one scalar pair per thread
        const long long bhp = (long long)bi * p.H + h_first + pre;
        cp_async4(lq + (pre % 3) * p.Q + tid, f.lcs + bhp * p.Lp + t0 + tid);
        cp_async4(dq + (pre % 3) * p.Q + tid, f.dte + bhp * p.Lp + t0 + tid);
      }
      cp_async_commit();
      const float Dcur = sD[hh];
      // one A_hat buffer: the MMAs of head hh-1 must have read it, so its
      // epilogue comes first; with two, the epilogue follows the mask pass
      if (!G.dbl && hh > 0) epilogue(hh - 1, li_prev, d_prev);
      uint8_t* sA = (G.dbl && buf) ? sA2 : sB;
      if (G.bal) {
        // Balanced mask pass (one column block, 128 rows).  Row block rb (32
        // rows) has 2 rb + 2 of its 16-column chunks on or below the diagonal,
        // so lane quarter 3 would carry 8 chunks and quarter 0 only 2.  Quarter
        // lo (0 or 1) therefore also takes the first 5 - (2 lo + 2) chunks of
        // its partner block hi = 3 - lo, read from C_rev B^T, whose lane quarter
        // lo holds the rows of block hi; every quarter does 5 chunks.  Chunks
        // wholly above the diagonal stay zero: they are written once per A_hat
        // buffer.
        const float* lb = lq + (hh % 3) * p.Q;
        const float* db = dq + (hh % 3) * p.Q;
        const int sq4 = wlane >> 5;
        const int lo = sq4 < 2 ? sq4 : 3 - sq4, hi = 3 - lo;
        const int nlo = 2 * lo + 2, split = 5 - nlo;
        for (int u = wg; u < 5; u += 4) {  // warp-uniform unit (row block, chunk)
          int rb, q;
          bool rev = false;
          if (sq4 == lo) {
            if (u < nlo) { rb = lo; q = u; }
            else { rb = hi; q = u - nlo; rev = true; }
          } else { rb = hi; q = split + u; }
          const int tok = rb * 32 + lane;
          const bool tok_ok = tok < len;
          const int st = tok_ok ? sq[tok] : -2;
          const float lt = tok_ok ? lb[tok] : 0.0f;
          uint32_t pk[8] = {0, 0, 0, 0, 0, 0, 0, 0};
          if (q * 16 < len) {
            float v[16];
            tmem_ld16(tmem_addr(rev ? tCB2 : tCB, wlane, q * 16), v);
            mask_unit(v, lb, db, sq, q * 16, tok_ok ? tok : -1, st, lt, one_seg, pk);
          }
          uint8_t* blk = sA + (q / 4) * (kRows * 128);
          const uint32_t e0 = (q % 4) * 16;
          *reinterpret_cast<uint4*>(blk + swz128_off(tok, e0)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
          *reinterpret_cast<uint4*>(blk + swz128_off(tok, e0 + 8)) = make_uint4(pk[4], pk[5], pk[6], pk[7]);
        }
        if (hh < 2)  // first use of this A_hat buffer: zero this quarter's chunks above the diagonal
          for (int q = 2 * sq4 + 2 + wg; q < 8; q += 4) {
            uint8_t* blk = sA + (q / 4) * (kRows * 128);
            const uint32_t e0 = (q % 4) * 16;
            *reinterpret_cast<uint4*>(blk + swz128_off(ri, e0)) = make_uint4(0, 0, 0, 0);
            *reinterpret_cast<uint4*>(blk + swz128_off(ri, e0 + 8)) = make_uint4(0, 0, 0, 0);
          }
      } else {  // mask pass: row ri, column quarter wg of every block J
        const float* lb = lq + (hh % 3) * p.Q;
        const float* db = dq + (hh % 3) * p.Q;
        const float li = row_ok ? lb[i] : 0.0f;
        const int warp_last_row = i0 + wlane + 31;  // last row of this warp
        for (int J = 0; J < nJ; ++J) {
          uint8_t* aJ = sA + J * bsp;
          for (int q = wg * 2; q < wg * 2 + 2; ++q) {
            uint32_t pk[8] = {0, 0, 0, 0, 0, 0, 0, 0};
            if (J * kRows + q * 16 <= warp_last_row && J * kRows + q * 16 < len) {  // else all masked
              float v[16];
              tmem_ld16(tmem_addr(tCB + J * 128, wlane, q * 16), v);
              mask_unit(v, lb, db, sq, J * kRows + q * 16, row_ok ? i : -1, si, li, one_seg, pk);
            }
            uint8_t* blk = aJ + (q / 4) * (kRows * 128);
            const uint32_t e0 = (q % 4) * 16;
            *reinterpret_cast<uint4*>(blk + swz128_off(ri, e0)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
            *reinterpret_cast<uint4*>(blk + swz128_off(ri, e0 + 8)) = make_uint4(pk[4], pk[5], pk[6], pk[7]);
          }
        }
      }
      const float li_hh = row_ok ? lq[(hh % 3) * p.Q + i] : 0.0f;  // before its slot can be refilled
      cp_async_wait_all();  // this thread's scalar copies have landed
      fence_async_smem();
      tc_fence_before();
      named_sync_compute();  // A_hat of head hh complete; every thread's copies of this iteration visible
      if (tid == 0) mbar_arrive(&b_ahat[buf]);
      if (G.dbl && hh > 0) epilogue(hh - 1, li_prev, d_prev);
      li_prev = li_hh;
      d_prev = Dcur;
    }
    epilogue(hpg - 1, li_prev, d_prev);
    if (lane == 0) bulk_wait_all();  // the tensor stores have finished before the block exits
  }
  if (!ok) atomicOr(&f.hdr->status, kDevTimeout);
  tc_fence_before();
  __syncthreads();
  if (tid < 32) tmem_dealloc(tm, 512);
}

}  // namespace

bool chunk_scan_tc_supported(const Plan& p) {
  return p.dtype == SSD_BF16 && p.P == 64 && (p.Q == 64 || p.Q == 128 || p.Q == 256) &&
         (p.N == 16 || p.N == 32 || p.N == 64 || p.N == 128) && p.hpg <= 256;
}

cudaError_t launch_chunk_scan_tc(const Plan& p, const Bufs& f, cudaStream_t s) {
  set_kernel_name("chunk_scan_tc");
  const ScanGeom G = scan_geom(p.N, p.Q);
  CUtensorMap tmC, tmB, tmX, tmH, tmC32, tmY;
  const uint32_t rows = (uint32_t)G.rows;
  const uint64_t dbc[4] = {(uint64_t)p.N, (uint64_t)p.G, (uint64_t)p.L, (uint64_t)p.b};
  const uint64_t sbc[3] = {(uint64_t)p.N * 2, (uint64_t)p.G * p.N * 2, (uint64_t)p.L * p.G * p.N * 2};
  const uint32_t bbc[4] = {(uint32_t)(G.cw / 2), 1, rows, 1};
  const uint32_t bbc32[4] = {(uint32_t)(G.cw / 2), 1, 32, 1};  // 32-row boxes for C_rev
  const uint64_t dxx[4] = {64, (uint64_t)p.H, (uint64_t)p.L, (uint64_t)p.b};
  const uint64_t sxx[3] = {128, (uint64_t)p.H * 128, (uint64_t)p.L * p.H * 128};
  const uint32_t bxx[4] = {64, 1, rows, 1};
  const uint32_t byy[4] = {16, 1, 32, 1};  // one warp's 32 rows x 16 columns of y, no swizzle
  // carry-in states (b*H, nc, N, 64) bf16
  const uint64_t dh[4] = {64, (uint64_t)p.N, (uint64_t)p.nc, (uint64_t)p.b * p.H};
  const uint64_t sh[3] = {128, (uint64_t)p.N * 128, (uint64_t)p.nc * p.N * 128};
  const uint32_t bh[4] = {64, (uint32_t)p.N, 1, 1};
  if (!encode_tmap_bf16_4d(&tmC, f.C, dbc, sbc, bbc, G.cw) ||
      !encode_tmap_bf16_4d(&tmB, f.B, dbc, sbc, bbc, G.cw) ||
      !encode_tmap_bf16_4d(&tmX, f.x, dxx, sxx, bxx, 128) ||
      !encode_tmap_bf16_4d(&tmH, f.Hin, dh, sh, bh, 128) ||
      !encode_tmap_bf16_4d(&tmC32, f.C, dbc, sbc, bbc32, G.cw) ||
      !encode_tmap_bf16_4d(&tmY, f.y, dxx, sxx, byy, 0))
    return cudaErrorInvalidValue;
  const size_t smem = 1024 + G.bytes + 7 * p.Q * 4 + 128 + (size_t)p.hpg * 4 + 16;
  cudaError_t e = cudaFuncSetAttribute(chunk_scan_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid(p.nc * G.nJ, p.G, p.b);
  chunk_scan_tc_kernel<<<grid, kThr, smem, s>>>(p, f, tmC, tmB, tmX, tmH, tmC32, tmY);
  return cudaGetLastError();
}

}  // namespace ssd
