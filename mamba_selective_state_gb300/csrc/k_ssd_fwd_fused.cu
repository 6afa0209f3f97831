// k_ssd_fwd_fused.cu -- the whole SSD forward in one persistent kernel.
//
// Page "llm-mamba-200" (gigipick.blogspot.com), kernel-fusion section and the
// "shared memory caching" section: the chunk's carry-out state is the next
// chunk's carry-in, so a kernel that walks a (batch row, head) chain in chunk
// order can keep the carry on chip and never write the chunk states.  One CTA
// owns one chain and, per chunk of kQ = 128 tokens:
//
//   dt_eff_j = softplus(dt_j + dt_bias_h),  l_i = sum_{k<=i} dt_eff_k A_h   (chunk-local)
//   [CB | Y2] = C [B ; H_in]^T                          (tensor cores, TMEM)
//   A_hat_ij = CB_ij exp(l_i - l_j) dt_eff_j  [j <= i, same sequence]
//   Y1       = A_hat X                                  (tensor cores)
//   y_i      = Y1_i + cv_i exp(l_i) Y2_i + D_h x_i
//   S^T      = B^T (w . X),  w_j = exp(l_last - l_j) dt_eff_j [seg_j = seg_last]
//   H_in     <- a_c H_in + S   (a_c = exp(l_last), 0 when a sequence starts in the chunk)
//
// with the carry H_in held in fp32 registers of the compute warps (one
// d_state row per TMEM lane, 16 headdim columns per thread) and handed to the
// tensor core as bf16 rows stacked under the B tile: C B^T and Y2 = C H_in^T
// share their A operand, so one N = 192 product forms both (a tcgen05.mma of
// N <= 128 costs about as much as one of N = 192).  The recurrence is the one of
// the chunked evaluation (page "llm-mamba-200", sections 1-3); the chunk
// length is internal to this kernel (the result does not depend on it).
//
// Warp roles (608 threads):
//   warps 0-15  compute: per chunk the carry update, the masked A_hat tile, the
//               weighted copy w . X of the next chunk and the y epilogue; warp w
//               reads TMEM lane quarter w % 4 (its SM sub-partition)
//   warp 16     control: one lane issues every TMA copy and every tcgen05.mma
//   warps 17-18 scalars: softplus, the chunk cumsum, decays and sequence
//               resets of the chunks ahead (even and odd chunks), into a ring
//               of three slots
// Lane quarter q holds rows 32q..32q+31 of the chunk and so the 2q+2
// 16-column units of A_hat on or below the diagonal.  Units strictly below
// the diagonal block of their 32-row block factor the decay as
// exp(l_i - l_r) exp(l_r - l_j) with l_r the l of the block's first row:
// both factors are <= 1 (l is nonincreasing when A_h <= 0), so the
// per-column factors are a table formed once per chunk and the unit needs
// two multiplies per entry instead of an exponential; the heavy quarters'
// extra units are of this kind, the two diagonal units of every quarter take
// the exact exponential.  (Shared-memory bandwidth, shared by the tensor
// core's operand reads and the warps, bounds this kernel: a second product
// to balance the quarters would cost more operand traffic than it saves.)
#include "ssd_internal.cuh"
#include "tc_common.cuh"
#include "tma_host.h"

namespace ssd {

namespace {

using namespace tc;

constexpr int kQ = 128;               // tokens per chunk = MMA M
constexpr int kCompute = 512;         // 16 compute warps
constexpr int kCtl = kCompute;        // first thread of the control warp
constexpr int kScal = kCompute + 32;  // first thread of the two scalar warps
constexpr int kThr = kCompute + 96;
constexpr int kRing = 3;              // scalar slots
constexpr int kXbuf = 3;              // x tiles (the epilogue stages y in them)

// One scalar slot: per token l, dt_eff, w, cve (= cv exp(l)), the factor
// tables s[rb-1][j] = exp(l_{32 rb} - l_j) dt_eff_j (j < 32 rb) of row blocks
// 1..3 and sd[j] = exp(l_{32 (j/32)} - l_j) dt_eff_j (j's own block), the
// segment ids, and per chunk a_c, one_seg, len, the two factoring flags and
// the reference l of each row block.
struct alignas(16) Slot {
  float l[kQ], dte[kQ], w[kQ], cve[kQ], s[3][kQ], sd[kQ];
  int sq[kQ];
  float a_c;
  int one_seg, len, fact, fact_diag;
  float lref[4];
};

struct FusedGeom {
  int ncb;          // 64-column blocks of B/C along d_state
  uint32_t cblk;    // bytes of one C column block (kQ rows x 128 B)
  uint32_t bhblk;   // bytes of one [B ; H_in] column block (kQ + 64 rows x 128 B)
  uint32_t offX, offB, offC, offXs, offA, offH, offSl, offBar, bytes;
};

__host__ __device__ inline FusedGeom fused_geom(int N) {
  FusedGeom g;
  g.ncb = N / 64;
  g.cblk = kQ * 128u;
  g.bhblk = (kQ + 64) * 128u;
  g.offX = 0;
  // [B ; H_in] blocks: the chunk's 128 B rows, then the 64 headdim rows of
  // the carry-in state (K = d_state in both)
  g.offB = g.offX + kXbuf * g.cblk;
  // with d_state 64 the product B^T (w . X) reads a second (unused) 64-row
  // block of A past the [B ; H_in] block: the C tile
  g.offC = g.offB + g.ncb * g.bhblk;
  g.offXs = g.offC + g.ncb * g.cblk;
  g.offA = g.offXs + g.cblk;
  // the carry-in state as a (d_state rows, 64 bf16) tile for the tensor
  // store of the kept intermediates
  g.offH = g.offA + 2u * g.cblk;
  g.offSl = g.offH + ((uint32_t)N * 128u + 1023u) / 1024u * 1024u;
  g.offBar = g.offSl + (uint32_t)(kRing * sizeof(Slot) + 255) / 256u * 256u;
  g.bytes = g.offBar + 256u;
  return g;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ uint32_t scale_bf16x2(uint32_t v, float w) {
  const float2 f = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&v));
  return pack_bf16x2(f.x * w, f.y * w);
}

__device__ __forceinline__ float softplus_f(float z) { return fmaxf(z, 0.0f) + log1pf(expf(-fabsf(z))); }

// Bounded wait; once a wait of this thread has failed, the later ones only
// spin briefly (the results are garbage by then, but the kernel still waits
// for the copies and products it issued before it exits).
__device__ __forceinline__ void wait_or_flag(uint64_t* bar, uint32_t parity, bool& ok) {
  if (ok) {
    if (!mbar_wait(bar, parity)) ok = false;
    return;
  }
  for (int i = 0; i < 4096; ++i)
    if (mbar_try_wait(bar, parity)) return;
}

// Exact unit: this thread's row `tok` against columns j0..j0+15:
// (C_tok . B_j) exp(l_tok - l_j) dt_j for j <= tok in the row's sequence, else 0.
__device__ __forceinline__ void unit_exact(const float (&v)[16], const Slot& S, int j0, int lim, int st,
                                           float lt, uint32_t (&pk)[8]) {
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float4 lj = *reinterpret_cast<const float4*>(S.l + j0 + 4 * k);
    const float4 dj = *reinterpret_cast<const float4*>(S.dte + j0 + 4 * k);
    int4 sj = make_int4(st, st, st, st);
    if (!S.one_seg) sj = *reinterpret_cast<const int4*>(S.sq + j0 + 4 * k);
    const float lv[4] = {lj.x, lj.y, lj.z, lj.w}, dv[4] = {dj.x, dj.y, dj.z, dj.w};
    const int sv[4] = {sj.x, sj.y, sj.z, sj.w};
    float a[4];
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      const bool on = j0 + 4 * k + m <= lim && sv[m] == st;
      a[m] = v[4 * k + m] * __expf(on ? lt - lv[m] : -INFINITY) * dv[m];
    }
    pk[2 * k] = pack_bf16x2(a[0], a[1]);
    pk[2 * k + 1] = pack_bf16x2(a[2], a[3]);
  }
}

// Factored unit (strictly below the row block's diagonal block, one sequence
// in the chunk): (C_tok . B_j) * r * s_j, r = exp(l_tok - l_ref).
__device__ __forceinline__ void unit_fact(const float (&v)[16], const float* s, int j0, float r,
                                          uint32_t (&pk)[8]) {
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float4 sj = *reinterpret_cast<const float4*>(s + j0 + 4 * k);
    pk[2 * k] = pack_bf16x2(v[4 * k] * sj.x * r, v[4 * k + 1] * sj.y * r);
    pk[2 * k + 1] = pack_bf16x2(v[4 * k + 2] * sj.z * r, v[4 * k + 3] * sj.w * r);
  }
}

// Factored unit inside the row block's own 32-column diagonal block (every
// block's decay range at most e^80, so sd_j = exp(l_r - l_j) dt_j stays
// finite): (C_tok . B_j) * r * sd_j for j <= tok, else 0.
__device__ __forceinline__ void unit_fact_diag(const float (&v)[16], const float* sd, int j0, int lim, float r,
                                               uint32_t (&pk)[8]) {
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float4 sj = *reinterpret_cast<const float4*>(sd + j0 + 4 * k);
    const float sv[4] = {sj.x, sj.y, sj.z, sj.w};
    float a[4];
#pragma unroll
    for (int m = 0; m < 4; ++m) a[m] = j0 + 4 * k + m <= lim ? v[4 * k + m] * sv[m] * r : 0.0f;
    pk[2 * k] = pack_bf16x2(a[0], a[1]);
    pk[2 * k + 1] = pack_bf16x2(a[2], a[3]);
  }
}

__global__ void __launch_bounds__(kThr, 1) ssd_fwd_fused_kernel(Plan p, Bufs f,
                                                                const __grid_constant__ CUtensorMap tmX,
                                                                const __grid_constant__ CUtensorMap tmB,
                                                                const __grid_constant__ CUtensorMap tmC,
                                                                const __grid_constant__ CUtensorMap tmY,
                                                                const __grid_constant__ CUtensorMap tmHin) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const FusedGeom G = fused_geom(p.N);
  const int bi = blockIdx.x / p.H, h = blockIdx.x % p.H;
  const int g = h / p.hpg;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nch = (p.L + kQ - 1) / kQ;
  uint8_t* sX = sm + G.offX;     // [kXbuf] x tiles; y is staged in place
  uint8_t* sB = sm + G.offB;     // [B ; H_in] blocks
  uint8_t* sC = sm + G.offC;
  uint8_t* sXs = sm + G.offXs;   // w . X
  uint8_t* sA = sm + G.offA;     // A_hat, two 64-column blocks
  uint8_t* sH = sm + G.offH;     // kept carry-in state (d_state rows, 64 bf16)
  Slot* ring = reinterpret_cast<Slot*>(sm + G.offSl);
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + G.offBar);
  uint64_t *b_x = bar, *b_bc = bar + 3, *b_hin = bar + 4, *b_xs = bar + 5, *b_m1 = bar + 6, *b_ahat = bar + 7,
           *b_y = bar + 8, *b_ystg = bar + 9, *b_full = bar + 10, *b_empty = bar + 13;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + 16);
  const long long bh = (long long)bi * p.H + h;
  // keep the intermediates the backward would recompute (dt_eff, chunk
  // cumsums, per-chunk decays, bf16 carry-in states) in the workspace
  const bool keep = (p.flags & SSD_KEEP_FWD_STATES) != 0;

  if (tid == kCtl) {
    for (int k = 0; k < 3; ++k) mbar_init(&b_x[k], 1);
    mbar_init(b_bc, 1);
    mbar_init(b_hin, kCompute / 32);
    mbar_init(b_xs, kCompute / 32);
    mbar_init(b_m1, 1);
    mbar_init(b_ahat, kCompute / 32);
    mbar_init(b_y, 1);
    mbar_init(b_ystg, kCompute / 32);
    for (int k = 0; k < kRing; ++k) {
      mbar_init(&b_full[k], 1);
      mbar_init(&b_empty[k], kCompute / 32);
    }
    mbar_fence_init();
    prefetch_tmap(&tmX);
    prefetch_tmap(&tmB);
    prefetch_tmap(&tmC);
    prefetch_tmap(&tmY);
  }
  if (warp == 0) tmem_alloc(tmem_slot, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tm = *tmem_slot;
  // [CB | Y2] double-buffered (2 x 192 columns) | S^T | Y1
  const uint32_t tCBY = tm, tS = tm + 384, tY1 = tm + 448;
  bool ok = true;

  if (warp == kCtl / 32) {
    // ------------------------------ control ------------------------------
    if (lane == 0) {
      const uint32_t xbytes = G.cblk;
      auto load_x = [&](int c) {
        const int k = c % kXbuf;
        mbar_expect_tx(&b_x[k], xbytes);
        tma_load_4d(sX + k * G.cblk, &tmX, &b_x[k], 0, h, c * kQ, bi);
      };
      auto load_bc = [&](int c) {
        mbar_expect_tx(b_bc, G.ncb * 2u * G.cblk);
        for (int q = 0; q < G.ncb; ++q) {
          tma_load_4d(sB + q * G.bhblk, &tmB, b_bc, q * 64, g, c * kQ, bi);
          tma_load_4d(sC + q * G.cblk, &tmC, b_bc, q * 64, g, c * kQ, bi);
        }
      };
      const uint32_t id192 = idesc_bf16(128, 192, 0, 0);  // K-major A and B
      const uint32_t id64b = idesc_bf16(128, 64, 0, 1);   // K-major A, MN-major B
      const uint32_t idS = idesc_bf16(128, 64, 1, 1);     // MN-major A and B
      load_x(0);
      if (nch > 1) load_x(1);
      if (nch > 2) load_x(2);
      load_bc(0);
      for (int c = 0; c < nch; ++c) {
        const uint32_t ph = c & 1;
        wait_or_flag(b_bc, ph, ok);
        wait_or_flag(b_hin, ph, ok);
        wait_or_flag(b_xs, ph, ok);
        tc_fence_after();
        if (keep) {  // the carry-in state of chunk c, as the products read it
          tma_store_4d(&tmHin, sH, 0, 0, c, (int)bh);
          bulk_commit();
        }
        // group 1: [C B^T | Y2 = C H_in^T], S^T = B^T (w . X)
        for (int ks = 0; ks < p.N / 16; ++ks) {
          const uint32_t kb = ks >> 2, kin = (ks & 3) * 32;
          const uint64_t dc = smem_desc(smem_u32(sC) + kb * G.cblk + kin, 16, 1024, kSwz128);
          const uint64_t dbh = smem_desc(smem_u32(sB) + kb * G.bhblk + kin, 16, 1024, kSwz128);
          mma_bf16(tCBY + ph * 192, dc, dbh, id192, ks > 0);
        }
        for (int ks = 0; ks < kQ / 16; ++ks) {
          const uint64_t da = smem_desc(smem_u32(sB) + ks * 2048, G.bhblk, 1024, kSwz128);
          const uint64_t dx = smem_desc(smem_u32(sXs) + ks * 2048, 16, 1024, kSwz128);
          mma_bf16(tS, da, dx, idS, ks > 0);
        }
        if (keep) bulk_wait_read<0>();  // the carry update of chunk c rewrites the tile
        mma_commit(b_m1);
        // y of the previous chunk: store it from its x tile, then refill
        // that tile with the chunk after next
        if (c >= 1) {
          wait_or_flag(b_ystg, (c - 1) & 1, ok);
          fence_async_smem();
          tma_store_4d(&tmY, sX + ((c - 1) % kXbuf) * G.cblk, 0, h, (c - 1) * kQ, bi);
          bulk_commit();
          if (c + 2 < nch) {
            bulk_wait_read<0>();
            load_x(c + 2);
          }
        }
        wait_or_flag(b_m1, ph, ok);  // B, C and w . X are free
        if (c + 1 < nch) load_bc(c + 1);
        wait_or_flag(b_ahat, ph, ok);
        tc_fence_after();
        const uint8_t* xt = sX + (c % kXbuf) * G.cblk;
        for (int ks = 0; ks < kQ / 16; ++ks) {  // Y1 = A_hat X
          const uint64_t da = smem_desc(smem_u32(sA) + (ks >> 2) * G.cblk + (ks & 3) * 32, 16, 1024, kSwz128);
          const uint64_t dx = smem_desc(smem_u32(xt) + ks * 2048, 16, 1024, kSwz128);
          mma_bf16(tY1, da, dx, id64b, ks > 0);
        }
        mma_commit(b_y);
      }
      wait_or_flag(b_ystg, (nch - 1) & 1, ok);
      fence_async_smem();
      tma_store_4d(&tmY, sX + ((nch - 1) % kXbuf) * G.cblk, 0, h, (nch - 1) * kQ, bi);
      bulk_commit();
      bulk_wait_all();
      wait_or_flag(b_y, (nch - 1) & 1, ok);  // the last products have completed
    }
  } else if (warp >= kScal / 32) {
    // ------------------------------ scalars ------------------------------
    const float bias = f.dt_bias[h], Ah = f.A[h];
    const bool fact_ok = Ah <= 0.0f;  // l nonincreasing: both factors of a split decay are <= 1
    const __nv_bfloat16* dtp = static_cast<const __nv_bfloat16*>(f.dt);
    const bool has_seq = f.seq != nullptr;
    const int* seqr = has_seq ? f.seq + (long long)bi * p.L : nullptr;
    auto load_raw = [&](int c, float (&raw)[4], int (&sg)[4]) {
      const int t0 = c * kQ;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int j = 4 * lane + k;
        raw[k] = 0.0f;
        sg[k] = -1;
        if (c < nch && t0 + j < p.L) {
          raw[k] = __bfloat162float(dtp[((long long)bi * p.L + t0 + j) * p.H + h]);
          if (has_seq) sg[k] = __ldg(seqr + t0 + j);
        }
      }
    };
    // scalar warp sw fills the slots of chunks sw, sw + 2, ...
    const int sw = warp - kScal / 32;
    float raw[4];
    int sg[4];
    load_raw(sw, raw, sg);
    for (int c = sw; c < nch; c += 2) {
      const int slot = c % kRing;
      float rawn[4];
      int sgn[4];
      load_raw(c + 2, rawn, sgn);  // this warp's next chunk: loads in flight during this one
      const int t0 = c * kQ, len = min(kQ, p.L - t0);
      float de[4], lv[4], run = 0.0f;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int j = 4 * lane + k;
        de[k] = j < len ? softplus_f(raw[k] + bias) : 0.0f;
        run += de[k] * Ah;
        lv[k] = run;
      }
      float incl = run;
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const float o = __shfl_up_sync(0xffffffffu, incl, d);
        if (lane >= d) incl += o;
      }
      float excl = __shfl_up_sync(0xffffffffu, incl, 1);
      if (lane == 0) excl = 0.0f;
#pragma unroll
      for (int k = 0; k < 4; ++k) lv[k] += excl;
      const float l_last = __shfl_sync(0xffffffffu, incl, 31);
      int seg_in = 0, seg_last = 0, seg_first = 0;
      if (has_seq) {
        seg_in = __ldg(seqr + (t0 > 0 ? t0 - 1 : 0));
        seg_last = __ldg(seqr + t0 + len - 1);
        seg_first = __ldg(seqr + t0);
      }
      float lref[4];
      bool diag_ok = true;  // every 32-token block spans a decay of e^80 or less
#pragma unroll
      for (int rb = 0; rb < 4; ++rb) {
        lref[rb] = __shfl_sync(0xffffffffu, lv[0], 8 * rb);
        diag_ok = diag_ok && (lref[rb] - __shfl_sync(0xffffffffu, lv[3], 8 * rb + 7) <= 80.0f);
      }
      if (c >= kRing) {
        bool okw = true;
        wait_or_flag(&b_empty[slot], ((c / kRing) - 1) & 1, okw);
        if (!okw) ok = false;
      }
      Slot& S = ring[slot];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int j = 4 * lane + k;
        const bool in = j < len;
        const int sj = has_seq ? sg[k] : 0;
        S.l[j] = lv[k];
        S.dte[j] = de[k];
        S.w[j] = (in && sj == seg_last) ? expf(l_last - lv[k]) * de[k] : 0.0f;
        S.cve[j] = (in && sj == seg_in) ? expf(lv[k]) : 0.0f;
        S.sq[j] = in ? sj : -1;
#pragma unroll
        for (int rb = 1; rb < 4; ++rb)
          S.s[rb - 1][j] = (in && j < 32 * rb) ? __expf(lref[rb] - lv[k]) * de[k] : 0.0f;
        S.sd[j] = (in && diag_ok) ? __expf(lref[lane >> 3] - lv[k]) * de[k] : 0.0f;
      }
      if (keep) {
        const long long base = bh * p.Lp + t0;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          f.dte[base + 4 * lane + k] = de[k];
          f.lcs[base + 4 * lane + k] = lv[k];
        }
      }
      if (lane == 0) {
        S.a_c = (seg_last == seg_in) ? expf(l_last) : 0.0f;
        if (keep) f.achunk[bh * p.nc + c] = S.a_c;
        S.one_seg = (seg_first == seg_last) ? 1 : 0;
        S.len = len;
        S.fact = (fact_ok && seg_first == seg_last) ? 1 : 0;
        S.fact_diag = (S.fact && diag_ok) ? 1 : 0;
#pragma unroll
        for (int rb = 0; rb < 4; ++rb) S.lref[rb] = lref[rb];
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&b_full[slot]);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        raw[k] = rawn[k];
        sg[k] = sgn[k];
      }
    }
  } else {
    // ------------------------------ compute ------------------------------
    const int sq4 = warp & 3, wg = warp >> 2;
    const int n = 32 * sq4 + lane;  // d_state row of the carry / output row of the chunk
    const int p0 = 16 * wg;         // headdim columns of this thread
    const bool nvalid = n < p.N;
    const bool hwarp = 32 * sq4 < p.N;  // warp-uniform: this warp holds carry rows
    const float Dh = f.D[h];
    float hreg[16];
#pragma unroll
    for (int k = 0; k < 16; ++k)
      hreg[k] = (f.init != nullptr && nvalid) ? f.init[(bh * p.P + p0 + k) * p.N + n] : 0.0f;
    // the carry as bf16 rows of the [B ; H_in] blocks: headdim row p, d_state
    // column n (K-major, like the B rows above it); with the forward's
    // intermediates kept, also as row n of the (d_state, headdim) tile that
    // the control lane stores
    auto write_h = [&]() {
      if (nvalid) {
        uint8_t* hb = sB + (n >> 6) * G.bhblk + kQ * 128u;
#pragma unroll
        for (int k = 0; k < 16; ++k)
          *reinterpret_cast<__nv_bfloat16*>(hb + swz128_off(p0 + k, n & 63)) = __float2bfloat16_rn(hreg[k]);
        if (keep) {
          uint32_t w8[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) w8[e] = pack_bf16x2(hreg[2 * e], hreg[2 * e + 1]);
          *reinterpret_cast<uint4*>(sH + swz128_off(n, p0)) = make_uint4(w8[0], w8[1], w8[2], w8[3]);
          *reinterpret_cast<uint4*>(sH + swz128_off(n, p0 + 8)) = make_uint4(w8[4], w8[5], w8[6], w8[7]);
        }
      }
    };
    auto arrive = [&](uint64_t* b) {
      __syncwarp();
      if (lane == 0) mbar_arrive(b);
    };
    // w . X of chunk c: warp w scales rows 8 w .. 8 w + 7, 8 lanes per
    // 128-byte row (conflict-free; the tile's swizzle permutes the 16-byte
    // pieces within a row, so the scaled copy keeps the layout)
    auto scale_x = [&](int c) {
      const Slot& S = ring[c % kRing];
      wait_or_flag(&b_full[c % kRing], (c / kRing) & 1, ok);
      wait_or_flag(&b_x[c % kXbuf], (c / kXbuf) & 1, ok);
      const uint4* src = reinterpret_cast<const uint4*>(sX + (c % kXbuf) * G.cblk);
      uint4* dst = reinterpret_cast<uint4*>(sXs);
#pragma unroll
      for (int it = 0; it < 2; ++it) {
        const int r = 8 * warp + 4 * it + (lane >> 3), e = r * 8 + (lane & 7);
        const float wr = S.w[r];
        uint4 v = src[e];
        v.x = scale_bf16x2(v.x, wr);
        v.y = scale_bf16x2(v.y, wr);
        v.z = scale_bf16x2(v.z, wr);
        v.w = scale_bf16x2(v.w, wr);
        dst[e] = v;
      }
      fence_async_smem();
      arrive(b_xs);
    };
    // prologue: initial carry, the A_hat zeros above the diagonal blocks,
    // w . X of chunk 0
    write_h();
    fence_async_smem();
    arrive(b_hin);
    for (int q = 2 * sq4 + 2 + wg; q < 8; q += 4) {
      uint8_t* blk = sA + (q >> 2) * G.cblk;
      const uint32_t e0 = (q & 3) * 16;
      *reinterpret_cast<uint4*>(blk + swz128_off(n, e0)) = make_uint4(0, 0, 0, 0);
      *reinterpret_cast<uint4*>(blk + swz128_off(n, e0 + 8)) = make_uint4(0, 0, 0, 0);
    }
    scale_x(0);
    for (int c = 0; c < nch; ++c) {
      const int slot = c % kRing;
      const Slot& S = ring[slot];
      wait_or_flag(b_m1, c & 1, ok);
      tc_fence_after();
      // ---- carry update: H_in[c+1] = a_c H_in[c] + S_c
      if (hwarp) {
        float sv[16];
        tmem_ld16(tmem_addr(tS, 32 * sq4, p0), sv);
        const float a = S.a_c;
#pragma unroll
        for (int k = 0; k < 16; ++k) hreg[k] = fmaf(a, hreg[k], sv[k]);
        if (c + 1 < nch) {
          write_h();
        } else if (f.final_states != nullptr && nvalid) {
#pragma unroll
          for (int k = 0; k < 16; ++k) f.final_states[(bh * p.P + p0 + k) * p.N + n] = hreg[k];
        }
      }
      fence_async_smem();
      tc_fence_before();
      arrive(b_hin);
      // ---- A_hat: row 32 sq4 + lane, the 2 sq4 + 2 units on or below the diagonal
      {
        const int len = S.len;
        const int tok = n;
        const bool tok_ok = tok < len;
        const float r_row = __expf(S.l[tok] - S.lref[sq4]);
        for (int q = wg; q <= 2 * sq4 + 1; q += 4) {
          uint32_t pk[8] = {0, 0, 0, 0, 0, 0, 0, 0};
          if (q * 16 < len) {  // warp-uniform
            float v[16];
            tmem_ld16(tmem_addr(tCBY + (c & 1) * 192, 32 * sq4, q * 16), v);
            if (S.fact && q < 2 * sq4) {
              unit_fact(v, S.s[sq4 - 1], q * 16, r_row, pk);
            } else if (S.fact_diag) {  // diagonal block, factored within it
              unit_fact_diag(v, S.sd, q * 16, tok_ok ? tok : -1, r_row, pk);
            } else {
              unit_exact(v, S, q * 16, tok_ok ? tok : -1, tok_ok ? S.sq[tok] : -2, S.l[tok], pk);
            }
          }
          uint8_t* blk = sA + (q >> 2) * G.cblk;
          const uint32_t e0 = (q & 3) * 16;
          *reinterpret_cast<uint4*>(blk + swz128_off(tok, e0)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
          *reinterpret_cast<uint4*>(blk + swz128_off(tok, e0 + 8)) = make_uint4(pk[4], pk[5], pk[6], pk[7]);
        }
      }
      fence_async_smem();
      tc_fence_before();
      arrive(b_ahat);
      // ---- w . X of the next chunk (the products of this chunk have read the
      // tile: the carry update above waited for them)
      if (c + 1 < nch) scale_x(c + 1);
      // ---- epilogue: y = Y1 + cv e^l Y2 + D x, staged in place of x
      wait_or_flag(b_y, c & 1, ok);
      tc_fence_after();
      {
        // the accumulator reads are in flight while the x row comes from
        // shared memory
        uint32_t ar[16], br[16];
        tmem_ld16_issue(tmem_addr(tY1, 32 * sq4, p0), ar);
        tmem_ld16_issue(tmem_addr(tCBY + (c & 1) * 192 + 128, 32 * sq4, p0), br);
        const float cv = S.cve[n];
        uint8_t* xt = sX + (c % kXbuf) * G.cblk;
        uint4* x0p = reinterpret_cast<uint4*>(xt + swz128_off(n, p0));
        uint4* x1p = reinterpret_cast<uint4*>(xt + swz128_off(n, p0 + 8));
        const uint4 x0 = *x0p, x1 = *x1p;
        tmem_ld_wait2(ar, br);
        float a[16], b[16];
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          a[k] = __uint_as_float(ar[k]);
          b[k] = __uint_as_float(br[k]);
        }
        const uint32_t xs[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
        uint32_t o[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float2 xf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&xs[e]));
          o[e] = pack_bf16x2(fmaf(Dh, xf.x, fmaf(cv, b[2 * e], a[2 * e])),
                             fmaf(Dh, xf.y, fmaf(cv, b[2 * e + 1], a[2 * e + 1])));
        }
        *x0p = make_uint4(o[0], o[1], o[2], o[3]);
        *x1p = make_uint4(o[4], o[5], o[6], o[7]);
      }
      fence_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(b_ystg);
        mbar_arrive(&b_empty[slot]);
      }
    }
  }
  if (!ok) atomicOr(&f.hdr->status, kDevTimeout);
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tm, 512);
}

}  // namespace

bool ssd_fwd_fused_supported(const Plan& p) {
  return p.dtype == SSD_BF16 && p.P == 64 && p.Q == kQ && (p.N == 64 || p.N == 128);
}

cudaError_t launch_ssd_fwd_fused(const Plan& p, const Bufs& f, cudaStream_t s) {
  set_kernel_name("ssd_fwd_fused");
  const FusedGeom G = fused_geom(p.N);
  CUtensorMap tmX, tmB, tmC, tmY, tmHin;
  const uint64_t dxx[4] = {64, (uint64_t)p.H, (uint64_t)p.L, (uint64_t)p.b};
  const uint64_t sxx[3] = {128, (uint64_t)p.H * 128, (uint64_t)p.L * p.H * 128};
  const uint32_t bxx[4] = {64, 1, (uint32_t)kQ, 1};
  const uint64_t dbc[4] = {(uint64_t)p.N, (uint64_t)p.G, (uint64_t)p.L, (uint64_t)p.b};
  const uint64_t sbc[3] = {(uint64_t)p.N * 2, (uint64_t)p.G * p.N * 2, (uint64_t)p.L * p.G * p.N * 2};
  const uint32_t bbc[4] = {64, 1, (uint32_t)kQ, 1};
  if (!encode_tmap_bf16_4d(&tmX, f.x, dxx, sxx, bxx, 128) ||
      !encode_tmap_bf16_4d(&tmB, f.B, dbc, sbc, bbc, 128) ||
      !encode_tmap_bf16_4d(&tmC, f.C, dbc, sbc, bbc, 128) ||
      !encode_tmap_bf16_4d(&tmY, f.y, dxx, sxx, bxx, 128))
    return cudaErrorInvalidValue;
  // kept carry-in states (b, H, nc, N, P) bf16: one (N x 64) tile per chunk
  if (p.flags & SSD_KEEP_FWD_STATES) {
    const uint64_t dhs[4] = {64, (uint64_t)p.N, (uint64_t)p.nc, (uint64_t)p.b * p.H};
    const uint64_t shs[3] = {128, (uint64_t)p.N * 128, (uint64_t)p.nc * p.N * 128};
    const uint32_t bhs[4] = {64, (uint32_t)p.N, 1, 1};
    if (!encode_tmap_bf16_4d(&tmHin, f.Hin, dhs, shs, bhs, 128)) return cudaErrorInvalidValue;
  } else {
    tmHin = tmY;  // unused
  }
  const size_t smem = 1024 + G.bytes;
  cudaError_t e = cudaFuncSetAttribute(ssd_fwd_fused_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  ssd_fwd_fused_kernel<<<p.b * p.H, kThr, smem, s>>>(p, f, tmX, tmB, tmC, tmY, tmHin);
  return cudaGetLastError();
}

}  // namespace ssd
