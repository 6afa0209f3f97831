// k_state_chain.cu -- the backward's state chains in one pass each, the
// chain value kept on chip.
//
// Page "llm-mamba-200" (gigipick.blogspot.com), "shared memory caching"
// section: a chunk's carry-out is the next chunk's carry-in.  The backward
// needs two chains over the chunks of every (batch row, head):
//
//   forward:  H_in[0] = init (or 0),  H_in[c+1] = a_c H_in[c] + S_c,
//             S_c[n][p]  = sum_j w_j B_j[n] x_j[p],   w_j = sv_j exp(l_last - l_j) dt_eff_j
//   reverse:  G = dfinal (or 0);  for c = nc-1 .. 0:
//               dS_c = G,  dL/da_c = <G, H_in[c]>,  G = dHloc_c + a_c G,
//             dHloc_c[n][p] = sum_i w_i C_i[n] dy_i[p],  w_i = cv_i exp(l_i),
//             dinit = G
//
// (the reverse is the same recurrence run right to left; page "B200 Helion
// Mamba-2" (aitrends.kr/articles/109906), section "Helion based B200 kernel
// redesign", names its state passing forward and backward).  Instead of
// writing every S_c / dHloc_c in fp32 and scanning them in a second kernel,
// one CTA walks one chain in chunk order: per chunk the tensor core forms
// S_c^T = T2^T (w . T1) (M = d_state, N = headdim, K = the chunk's tokens;
// T1 = x or dy, T2 = B or C, both by TMA), and the compute warps fold it into
// the chain value held in fp32 registers (one d_state row per TMEM lane, 16
// headdim columns per thread), writing H_in[c] (forward) or dS_c (reverse)
// as the bf16 operands of the chunk-backward kernels.  dL/da_c is a fixed
// fold: per-warp sums (xor shuffles) into 16 slots per chunk, added in slot
// order by the parameter-gradient kernel.
//
// Warps: 16 compute (warp w reads TMEM lane quarter w % 4), 1 control (TMA
// and tcgen05.mma from one lane).  Three stages (T1, T2 and the chunk's l and
// dt_eff), two w . T1 tiles, two accumulators: the product of chunk k+1 runs
// while chunk k is folded.  The reverse chain's carry-in tiles (for dL/da_c)
// come by tensor copies into two buffers, each issued about two steps before
// its step reads it.
#include "ssd_internal.cuh"
#include "tc_common.cuh"
#include "tma_host.h"

namespace ssd {

namespace {

using namespace tc;

constexpr int kQ = 128;
constexpr int kCompute = 512;
constexpr int kThr = kCompute + 32;
constexpr int kStages = 3;

struct ChainGeom {
  int ncb;           // 64-column blocks of B/C along d_state
  uint32_t blk;      // bytes of one 128-row x 128-byte tile block
  uint32_t offScal;  // l and dt_eff of the stage's chunk (Q floats each), after its tiles
  uint32_t stage;    // T1 block + ncb T2 blocks + the scalars
  uint32_t hbytes;   // one carry-in tile (N rows of 64 bf16), reverse chain only
  uint32_t offXs, offH, offBar, bytes;
};

__host__ __device__ inline ChainGeom chain_geom(int N, bool rev) {
  ChainGeom g;
  g.ncb = N / 64;
  g.blk = kQ * 128u;
  g.offScal = g.blk * (1u + g.ncb);
  g.stage = g.offScal + 2u * kQ * 4u;  // a multiple of 1024
  // with d_state 64 the product reads a second (unused) 64-row column block
  // past T2: the scalars and the next stage's T1, or for the last stage the
  // w . T1 tiles
  g.hbytes = rev ? (uint32_t)N * 128u : 0u;
  g.offXs = kStages * g.stage;
  g.offH = g.offXs + 2u * g.blk;
  g.offBar = g.offH + 2u * g.hbytes;
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

__device__ __forceinline__ void wait_or_flag(uint64_t* bar, uint32_t parity, bool& ok) {
  if (ok) {
    if (!mbar_wait(bar, parity)) ok = false;
    return;
  }
  for (int i = 0; i < 4096; ++i)
    if (mbar_try_wait(bar, parity)) return;
}

template <bool kRev>
__global__ void __launch_bounds__(kThr, 1) state_chain_kernel(Plan p, Bufs f,
                                                              const __grid_constant__ CUtensorMap tm1,
                                                              const __grid_constant__ CUtensorMap tm2,
                                                              const __grid_constant__ CUtensorMap tmH) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const ChainGeom G = chain_geom(p.N, kRev);
  const int bi = blockIdx.x / p.H, h = blockIdx.x % p.H;
  const int g = h / p.hpg;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nc = p.nc;
  const long long bh = (long long)bi * p.H + h;
  uint8_t* sXs = sm + G.offXs;
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + G.offBar);
  uint8_t* sH = sm + G.offH;  // [2] carry-in tiles (reverse), 128-byte swizzled rows
  uint64_t *b_ld = bar, *b_xs = bar + kStages, *b_full = b_xs + 2, *b_free = b_full + 2, *b_done = b_free + 2,
           *b_h = b_done + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(b_h + 2);
  auto chunk_of = [&](int k) { return kRev ? nc - 1 - k : k; };

  if (tid == kCompute) {
    for (int k = 0; k < kStages; ++k) mbar_init(&b_ld[k], 1);
    for (int k = 0; k < 2; ++k) {
      mbar_init(&b_xs[k], kCompute / 32);
      mbar_init(&b_full[k], 1);
      mbar_init(&b_free[k], kCompute / 32);
    }
    mbar_init(b_done, 1);
    mbar_init(&b_h[0], 1);
    mbar_init(&b_h[1], 1);
    mbar_fence_init();
    prefetch_tmap(&tm1);
    prefetch_tmap(&tm2);
  }
  if (warp == 0) tmem_alloc(tmem_slot, 128);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tm = *tmem_slot;
  bool ok = true;

  if (warp == kCompute / 32) {
    // ------------------------------ control ------------------------------
    if (lane == 0) {
      // the stage of step k: T1, T2 and the chunk's l and dt_eff
      auto load = [&](int k) {
        const int s = k % kStages, c = chunk_of(k);
        uint8_t* st = sm + s * G.stage;
        mbar_expect_tx(&b_ld[s], G.stage);
        tma_load_4d(st, &tm1, &b_ld[s], 0, h, c * kQ, bi);
        for (int q = 0; q < G.ncb; ++q)
          tma_load_4d(st + (1 + q) * G.blk, &tm2, &b_ld[s], q * 64, g, c * kQ, bi);
        bulk_load(st + G.offScal, f.lcs + bh * p.Lp + (long long)c * kQ, kQ * 4, &b_ld[s]);
        bulk_load(st + G.offScal + kQ * 4, f.dte + bh * p.Lp + (long long)c * kQ, kQ * 4, &b_ld[s]);
      };
      // reverse: the carry-in tile of step k, for dL/da_c
      auto load_hin = [&](int k) {
        mbar_expect_tx(&b_h[k & 1], G.hbytes);
        tma_load_4d(sH + (k & 1) * G.hbytes, &tmH, &b_h[k & 1], 0, 0, chunk_of(k), (int)bh);
      };
      const uint32_t idS = idesc_bf16(128, 64, 1, 1);
      for (int k = 0; k < kStages && k < nc; ++k) load(k);
      if (kRev) load_hin(0);
      for (int k = 0; k < nc; ++k) {
        const int s = k % kStages, b = k & 1;
        wait_or_flag(&b_xs[b], (k >> 1) & 1, ok);
        if (k >= 2) wait_or_flag(&b_free[b], ((k - 2) >> 1) & 1, ok);
        tc_fence_after();
        const uint8_t* t2 = sm + s * G.stage + G.blk;
        const uint8_t* xs = sXs + b * G.blk;
        for (int ks = 0; ks < kQ / 16; ++ks) {
          const uint64_t da = smem_desc(smem_u32(t2) + ks * 2048, G.blk, 1024, kSwz128);
          const uint64_t db = smem_desc(smem_u32(xs) + ks * 2048, 16, 1024, kSwz128);
          mma_bf16(tm + b * 64, da, db, idS, ks > 0);
        }
        mma_commit(&b_full[b]);
        mma_commit(b_done);
        // the stage is free once this product has read it (w . T1 was read
        // from it before the compute warps signalled)
        wait_or_flag(b_done, k & 1, ok);
        if (k + kStages < nc) load(k + kStages);
        // the carry-in tile of step k+1 goes where step k-1's was, once that
        // step is done (about two steps before step k+1 reads it)
        if (kRev && k + 1 < nc) {
          if (k >= 1) wait_or_flag(&b_free[(k - 1) & 1], ((k - 1) >> 1) & 1, ok);
          load_hin(k + 1);
        }
      }
    }
  } else {
    // ------------------------------ compute ------------------------------
    const int sq4 = warp & 3, wg = warp >> 2;
    const int n = 32 * sq4 + lane;  // d_state row
    const int p0 = 16 * wg;         // headdim columns
    const bool nvalid = n < p.N;
    const bool hwarp = 32 * sq4 < p.N;  // warp-uniform
    const int* seqr = f.seq != nullptr ? f.seq + (long long)bi * p.L : nullptr;
    float v[16];
    {
      const float* src = kRev ? f.dfinal : f.init;
#pragma unroll
      for (int k = 0; k < 16; ++k) v[k] = (src != nullptr && nvalid) ? src[(bh * p.P + p0 + k) * p.N + n] : 0.0f;
    }
    // Per-step values loaded two steps ahead (their latency hides behind two
    // chunks of work): the chunk's decay and, with seq_idx, the segment ids
    // that decide this thread's row weight.  (The loads are unconditional,
    // from clamped addresses, so that they can land in the registers that
    // use them; the conditions apply at the use.)
    struct Raw {
      float a;  // the chunk's decay a_c
      int s, sref;
    };
    auto ld_raw = [&](int k) {
      Raw r;
      const int kk = k < nc ? k : nc - 1;
      const int c = chunk_of(kk), t0 = c * kQ, len = min(kQ, p.L - t0), row = tid >> 2;
      const int rr = row < len ? row : len - 1;
      r.a = __ldg(f.achunk + bh * nc + c);
      r.s = seqr ? __ldg(seqr + t0 + rr) : 0;
      r.sref = seqr ? __ldg(seqr + (kRev ? (t0 > 0 ? t0 - 1 : 0) : t0 + len - 1)) : 0;
      return r;
    };
    // w . T1 of step k: thread -> row tid/4, two 16-byte pieces (the tile's
    // swizzle permutes pieces within a row, so the scaled copy keeps it); the
    // row weight from the chunk's l and dt_eff that came with the stage
    auto scale = [&](int k, const Raw& r) {
      const int s = k % kStages;
      const int row = tid >> 2, part = tid & 3;
      wait_or_flag(&b_ld[s], (k / kStages) & 1, ok);
      const uint8_t* st = sm + s * G.stage;
      const float* sl = reinterpret_cast<const float*>(st + G.offScal);
      const int c = chunk_of(k), len = min(kQ, p.L - c * kQ);
      float wv = 0.0f;
      if (row < len && r.s == r.sref)
        wv = kRev ? expf(sl[row]) : expf(sl[len - 1] - sl[row]) * sl[kQ + row];
      const uint4* src = reinterpret_cast<const uint4*>(st + row * 128) + part * 2;
      uint4* dst = reinterpret_cast<uint4*>(sXs + (k & 1) * G.blk + row * 128) + part * 2;
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        uint4 t = src[q];
        t.x = scale_bf16x2(t.x, wv);
        t.y = scale_bf16x2(t.y, wv);
        t.z = scale_bf16x2(t.z, wv);
        t.w = scale_bf16x2(t.w, wv);
        dst[q] = t;
      }
      fence_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&b_xs[k & 1]);
    };
    // One step: chunk k's value is written out and the product of chunk k
    // folded in, while w . T1 of chunk k+1 is formed and the operands of the
    // steps ahead are in flight.  The prefetched registers ping-pong between
    // two sets (r_use read here, r_fill loaded here and read a step later),
    // so no copy waits on a load still in flight.
    auto step = [&](int k, Raw& r_fill, const Raw& r_use) {
      const float a = r_fill.a;  // a_c of chunk k, loaded two steps ago (before the set is refilled)
      r_fill = ld_raw(k + 2);
      if (k + 1 < nc) scale(k + 1, r_use);
      const int c = chunk_of(k), b = k & 1;
      __nv_bfloat16* out = static_cast<__nv_bfloat16*>(kRev ? f.dS : f.Hin) + ((bh * nc + c) * p.N + n) * 64 + p0;
      float dpart = 0.0f;
      if (hwarp && nvalid) {
        uint32_t w8[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) w8[e] = pack_bf16x2(v[2 * e], v[2 * e + 1]);
        reinterpret_cast<uint4*>(out)[0] = make_uint4(w8[0], w8[1], w8[2], w8[3]);
        reinterpret_cast<uint4*>(out)[1] = make_uint4(w8[4], w8[5], w8[6], w8[7]);
        if (kRev) {  // dL/da_c partial: <G, H_in[c]> over this thread's 16 entries
          wait_or_flag(&b_h[b], (k >> 1) & 1, ok);
          // row n of the tile, 16-byte pieces 2 wg and 2 wg + 1 (128-byte swizzle)
          const uint8_t* hrow = sH + b * G.hbytes + n * 128;
          const uint4 h0 = *reinterpret_cast<const uint4*>(hrow + (((2 * wg) ^ (n & 7)) << 4));
          const uint4 h1 = *reinterpret_cast<const uint4*>(hrow + (((2 * wg + 1) ^ (n & 7)) << 4));
          const uint32_t hw[8] = {h0.x, h0.y, h0.z, h0.w, h1.x, h1.y, h1.z, h1.w};
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const float2 hf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&hw[e]));
            dpart = fmaf(v[2 * e], hf.x, fmaf(v[2 * e + 1], hf.y, dpart));
          }
        }
      }
      if (kRev) {
#pragma unroll
        for (int d = 16; d > 0; d >>= 1) dpart += __shfl_xor_sync(0xffffffffu, dpart, d);
        if (lane == 0) f.dapart[((size_t)bh * nc + c) * p.da_stride + warp] = dpart;
      }
      wait_or_flag(&b_full[b], (k >> 1) & 1, ok);
      tc_fence_after();
      if (hwarp) {
        float sv[16];
        tmem_ld16(tmem_addr(tm + b * 64, 32 * sq4, p0), sv);
#pragma unroll
        for (int e = 0; e < 16; ++e) v[e] = fmaf(a, v[e], sv[e]);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&b_free[b]);
    };
    // set j & 1 holds the operands of chunk j
    Raw r0 = ld_raw(0), r1 = ld_raw(1);
    scale(0, r0);
    for (int k = 0; k < nc; k += 2) {
      step(k, r0, r1);
      if (k + 1 < nc) step(k + 1, r1, r0);
    }
    if (kRev && f.dinit != nullptr && nvalid) {
#pragma unroll
      for (int k = 0; k < 16; ++k) f.dinit[(bh * p.P + p0 + k) * p.N + n] = v[k];
    }
  }
  if (!ok) atomicOr(&f.hdr->status, kDevTimeout);
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tm, 128);
}

}  // namespace

bool state_chain_supported(const Plan& p) {
  return p.dtype == SSD_BF16 && p.P == 64 && p.Q == kQ && (p.N == 64 || p.N == 128) &&
         p.da_stride >= kCompute / 32;
}

cudaError_t launch_state_chain(const Plan& p, const Bufs& f, bool reverse, cudaStream_t s) {
  set_kernel_name(reverse ? "state_chain_bwd" : "state_chain_fwd");
  const ChainGeom G = chain_geom(p.N, reverse);
  CUtensorMap tm1, tm2, tmH;
  const uint64_t d1[4] = {64, (uint64_t)p.H, (uint64_t)p.L, (uint64_t)p.b};
  const uint64_t s1[3] = {128, (uint64_t)p.H * 128, (uint64_t)p.L * p.H * 128};
  const uint32_t b1[4] = {64, 1, (uint32_t)kQ, 1};
  const uint64_t d2[4] = {(uint64_t)p.N, (uint64_t)p.G, (uint64_t)p.L, (uint64_t)p.b};
  const uint64_t s2[3] = {(uint64_t)p.N * 2, (uint64_t)p.G * p.N * 2, (uint64_t)p.L * p.G * p.N * 2};
  const uint32_t b2[4] = {64, 1, (uint32_t)kQ, 1};
  // carry-in states (b, H, nc, N, P) bf16: one chunk's N x 64 tile per copy
  const uint64_t dh[4] = {64, (uint64_t)p.N, (uint64_t)p.nc, (uint64_t)p.b * p.H};
  const uint64_t sh[3] = {128, (uint64_t)p.N * 128, (uint64_t)p.nc * p.N * 128};
  const uint32_t bh[4] = {64, (uint32_t)p.N, 1, 1};
  if (!encode_tmap_bf16_4d(&tm1, reverse ? f.dy : f.x, d1, s1, b1, 128) ||
      !encode_tmap_bf16_4d(&tm2, reverse ? f.C : f.B, d2, s2, b2, 128))
    return cudaErrorInvalidValue;
  if (reverse) {
    if (!encode_tmap_bf16_4d(&tmH, f.Hin, dh, sh, bh, 128)) return cudaErrorInvalidValue;
  } else {
    tmH = tm1;  // not read by the forward chain
  }
  const size_t smem = 1024 + G.bytes;
  auto kern = reverse ? state_chain_kernel<true> : state_chain_kernel<false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  kern<<<p.b * p.H, kThr, smem, s>>>(p, f, tm1, tm2, tmH);
  return cudaGetLastError();
}

}  // namespace ssd
