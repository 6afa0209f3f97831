// k_chunk_bwd_tc.cu -- token gradients of one chunk on the 5th-generation
// tensor cores (reverse mode of the chunk output and the chunk state).
//
// Notation (chunk c, head h, chunk-local tokens i, j):
//   E_ij = exp(l_i - l_j) [j <= i, seg_i = seg_j],  M_ij = (C_i.B_j) E_ij dt_j,
//   dM_ij = dy_i . x_j,  u_j = sv_j exp(l_last - l_j) dt_j,  dS = dL/dS_c,
//   H = carry-in state of the chunk.
//
// chunk_bwd_tc (one CTA per row, chunk, head) writes
//   dx_j      = sum_{i>=j} M_ij dy_i + u_j dS B_j + D_h dy_j
//   ddt_eff_j = sum_{i>=j} dM_ij (C_i.B_j) E_ij + sv_j exp(l_last-l_j) (x_j.dS B_j)
//   dl_t      = sum_j dM_tj M_tj - sum_i dM_it M_it + [cv_t] e^{l_t} dy_t.(H C_t) - u_t (x_t.dS B_t)
// and per-chunk partials sum_j u_j (x_j.dS B_j), sum dy.x.  Every
// 128 x 128 token tile is formed in both orientations on the tensor cores
// (C B^T and B C^T, dy x^T and x dy^T), so each row sum and each column sum
// is taken by the thread that owns that token, in fp32 and in a fixed order.
//
// chunk_bwd_dbc_tc (one CTA per row, chunk, group, 128-token block T) writes
//   dC_i = sum_h [ sum_{j<=i} dM_ij E_ij dt_j B_j + cv_i e^{l_i} H^T dy_i ]     (i in T)
//   dB_j = sum_h [ sum_{i>=j} dM_ij E_ij dt_j C_i + u_j dS^T x_j ]            (j in T)
// accumulating both in tensor memory over the heads of the group in a fixed
// order (no atomics: bitwise reproducible).
// Operands arrive by TMA; derived operands (masked tiles, row-scaled copies)
// are written to shared memory by the four warps as K-major bf16 tiles.
#include "ssd_internal.cuh"
#include "tc_common.cuh"
#include "tma_host.h"

namespace ssd {

namespace {

using namespace tc;

constexpr int kRows = 128;
constexpr int kThr = 128;

__host__ __device__ inline uint32_t r1024(uint32_t v) { return (v + 1023u) & ~1023u; }

struct Tiles {
  int rows;        // rows per token TMA box = min(Q, 128)
  int cw, ncb;     // bytes per row of a B/C column block, column blocks
  uint32_t cblk;   // bytes of one B/C column block (128 rows)
  uint32_t cswz;   // swizzle code of B/C tiles
  uint32_t cbytes; // bytes of one B or C tile
  uint32_t sbytes; // bytes of one (N x 64) state tile (dS or H)
};

__host__ __device__ inline Tiles tiles(int N, int Q) {
  Tiles t;
  t.rows = Q < kRows ? Q : kRows;
  t.cw = 2 * (N < 64 ? N : 64);
  t.ncb = N >= 64 ? N / 64 : 1;
  t.cblk = (uint32_t)kRows * t.cw;
  t.cswz = t.cw == 128 ? kSwz128 : (t.cw == 64 ? kSwz64 : kSwz32);
  t.cbytes = r1024(t.ncb * t.cblk);
  t.sbytes = r1024((uint32_t)N * 128u);
  return t;
}

constexpr uint32_t kTok = kRows * 128u;  // one (128 tokens x 64) bf16 tile
constexpr uint32_t kAhat = 2u * kRows * 128u;  // 128 x 128 bf16, two K blocks

__device__ __forceinline__ uint32_t pack2(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}
__device__ __forceinline__ float2 unpack2(uint32_t v) {
  return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&v));
}

// K-major A (or B) descriptor of k-step ks of a B/C tile (K = d_state)
__device__ __forceinline__ uint64_t desc_c_kmajor(const Tiles& T, const uint8_t* t, int ks) {
  const uint32_t kb = (ks * 32) / T.cw, kin = (ks * 32) % T.cw;
  return smem_desc(smem_u32(t) + kb * T.cblk + kin, 16, 8 * T.cw, T.cswz);
}
// MN-major B descriptor of k-step ks of a B/C tile used with K = tokens
__device__ __forceinline__ uint64_t desc_c_mnmajor(const Tiles& T, const uint8_t* t, int ks) {
  return smem_desc(smem_u32(t) + ks * 16 * T.cw, T.cblk, 8 * T.cw, T.cswz);
}
// K-major descriptor of a 128 x 64 token tile (K = headdim) or of A_hat
__device__ __forceinline__ uint64_t desc_tok_kmajor(const uint8_t* t, int ks) {
  return smem_desc(smem_u32(t) + (ks / 4) * kTok + (ks % 4) * 32, 16, 1024, kSwz128);
}
// MN-major descriptor of a 128 x 64 token tile (K = tokens) or of an N x 64 state tile (K = d_state)
__device__ __forceinline__ uint64_t desc_rows_mnmajor(const uint8_t* t, int ks) {
  return smem_desc(smem_u32(t) + ks * 16 * 128, 16, 1024, kSwz128);
}

__device__ __forceinline__ bool wait_mma(uint64_t* bar, uint32_t& ph) {
  const bool r = mbar_wait(bar, ph);
  ph ^= 1;
  tc_fence_after();
  return r;
}

// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kThr) chunk_bwd_tc_kernel(Plan p, Bufs f,
                                                            const __grid_constant__ CUtensorMap tmX,
                                                            const __grid_constant__ CUtensorMap tmY,
                                                            const __grid_constant__ CUtensorMap tmB,
                                                            const __grid_constant__ CUtensorMap tmC,
                                                            const __grid_constant__ CUtensorMap tmS,
                                                            const __grid_constant__ CUtensorMap tmH) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const Tiles T = tiles(p.N, p.Q);
  uint8_t* sX = sm;
  uint8_t* sY = sX + kTok;
  uint8_t* sB = sY + kTok;
  uint8_t* sC = sB + T.cbytes;
  const bool alias = T.cbytes >= kAhat;
  uint8_t* sA = alias ? sC : sC + T.cbytes;
  uint8_t* sS = alias ? sC + T.cbytes : sA + kAhat;
  uint8_t* sH = sS + T.sbytes;
  float* lq = reinterpret_cast<float*>(sH + T.sbytes);
  float* dq = lq + p.Q;
  float* dda = dq + p.Q;
  float* dla = dda + p.Q;
  int* sq = reinterpret_cast<int*>(dla + p.Q);
  float* red = reinterpret_cast<float*>(sq + p.Q);  // 3 x kThr
  uint64_t* bar = reinterpret_cast<uint64_t*>(red + 3 * kThr);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + 2);

  const int c = blockIdx.x, h = blockIdx.y, bi = blockIdx.z;
  const int g = h / p.hpg;
  const int tid = threadIdx.x, wlane = (tid >> 5) * 32;
  const int t0 = c * p.Q, len = min(p.Q, p.L - t0);
  const long long bh = (long long)bi * p.H + h;
  const int nb = (p.Q + kRows - 1) / kRows;

  for (int t = tid; t < p.Q; t += kThr) {
    lq[t] = f.lcs[bh * p.Lp + t0 + t];
    dq[t] = f.dte[bh * p.Lp + t0 + t];
    sq[t] = t < len ? seg_of(p, f, bi, (long long)t0 + t) : -1;
    dda[t] = 0.0f;
    dla[t] = 0.0f;
  }
  if (T.rows < kRows)  // K padding of the token-contracted MMAs must be zero
    for (int idx = tid; idx < (kRows - T.rows) * 8; idx += kThr) {
      reinterpret_cast<uint4*>(sX + T.rows * 128)[idx] = make_uint4(0, 0, 0, 0);
      reinterpret_cast<uint4*>(sY + T.rows * 128)[idx] = make_uint4(0, 0, 0, 0);
    }
  if (tid == 0) {
    mbar_init(&bar[0], 1);
    mbar_init(&bar[1], 1);
    mbar_fence_init();
  }
  if (tid < 32) tmem_alloc(tmem_slot, 512);
  fence_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tm = *tmem_slot;
  const uint32_t tT0 = tm, tT1 = tm + 128, tDX = tm + 256, tDXS = tm + 320, tYC = tm + 384;
  const int s_in = seg_in_of(p, f, bi, c);
  const int s_last = seg_of(p, f, bi, (long long)t0 + len - 1);
  const float l_last = lq[len - 1];
  const float Dh = f.D[h];
  bool ok = true;
  uint32_t ph_ld = 0, ph_mma = 0;
  float udu_part = 0.0f, dD_part = 0.0f;
  const uint32_t tok_bytes = (uint32_t)T.rows * 128u;
  const uint32_t c_bytes = (uint32_t)T.ncb * T.rows * T.cw;

  if (tid == 0) {  // state tiles: loaded once
    mbar_expect_tx(&bar[0], 2u * (uint32_t)p.N * 128u);
    tma_load_4d(sS, &tmS, &bar[0], 0, 0, c, (int)bh);
    tma_load_4d(sH, &tmH, &bar[0], 0, 0, c, (int)bh);
  }
  if (!mbar_wait(&bar[0], ph_ld)) ok = false;
  ph_ld ^= 1;

  for (int J = 0; J < nb; ++J) {
    if (J * kRows >= len) break;
    bool first = true;
    for (int I = nb - 1; I >= J; --I) {
      if (I * kRows >= len) continue;
      const bool diag = (I == J);
      // every thread has finished its waits on both barriers' previous phases
      // before thread 0 arms them again; its shared reads of the tiles come
      // before the tensor copies that overwrite them
      tc_fence_before();
      fence_async_smem();
      __syncthreads();
      if (tid == 0) {
        mbar_expect_tx(&bar[0], 2 * tok_bytes + 2 * c_bytes);
        tma_load_4d(sX, &tmX, &bar[0], 0, h, t0 + J * kRows, bi);
        tma_load_4d(sY, &tmY, &bar[0], 0, h, t0 + I * kRows, bi);
        for (int q = 0; q < T.ncb; ++q) {
          tma_load_4d(sB + q * T.cblk, &tmB, &bar[0], q * 64, g, t0 + J * kRows, bi);
          tma_load_4d(sC + q * T.cblk, &tmC, &bar[0], q * 64, g, t0 + I * kRows, bi);
        }
      }
      if (!mbar_wait(&bar[0], ph_ld)) ok = false;
      ph_ld ^= 1;
      // ---- batch 1: row orientation (M = i) + diagonal extras
      if (tid == 0) {
        tc_fence_after();
        const uint32_t id128 = idesc_bf16(128, 128, 0, 0), id64 = idesc_bf16(128, 64, 0, 1);
        for (int ks = 0; ks < p.N / 16; ++ks)
          mma_bf16(tT0, desc_c_kmajor(T, sC, ks), desc_c_kmajor(T, sB, ks), id128, ks > 0);
        for (int ks = 0; ks < 4; ++ks)
          mma_bf16(tT1, desc_tok_kmajor(sY, ks), desc_tok_kmajor(sX, ks), id128, ks > 0);
        if (diag) {
          for (int ks = 0; ks < p.N / 16; ++ks) {
            mma_bf16(tYC, desc_c_kmajor(T, sC, ks), desc_rows_mnmajor(sH, ks), id64, ks > 0);
            mma_bf16(tDXS, desc_c_kmajor(T, sB, ks), desc_rows_mnmajor(sS, ks), id64, ks > 0);
          }
        }
        mma_commit(&bar[1]);
      }
      if (!wait_mma(&bar[1], ph_mma)) ok = false;
      {  // row pass: thread owns token i
        const int i = I * kRows + tid;
        const bool rok = i < len;
        const float li = rok ? lq[i] : 0.0f;
        const int si = rok ? sq[i] : -2;
        float acc = 0.0f;
        for (int q = 0; q < kRows / 16; ++q) {
          float cb[16], dm[16];
          tmem_ld16(tmem_addr(tT0, wlane, q * 16), cb);
          tmem_ld16(tmem_addr(tT1, wlane, q * 16), dm);
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const int j = J * kRows + q * 16 + e;
            if (rok && j <= i && sq[j] == si) acc += dm[e] * cb[e] * __expf(li - lq[j]) * dq[j];
          }
        }
        if (diag) {
          float s = 0.0f;
          for (int q = 0; q < 4; ++q) {
            float yc[16];
            tmem_ld16(tmem_addr(tYC, wlane, q * 16), yc);
            const uint4 a = *reinterpret_cast<const uint4*>(sY + swz128_off(tid, q * 16));
            const uint4 b = *reinterpret_cast<const uint4*>(sY + swz128_off(tid, q * 16 + 8));
            const uint32_t dy[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              const float2 d = unpack2(dy[e]);
              s += d.x * yc[2 * e] + d.y * yc[2 * e + 1];
            }
          }
          if (rok && si == s_in) acc += __expf(li) * s;
        }
        if (rok) dla[i] += acc;
      }
      tc_fence_before();
      __syncthreads();
      // ---- batch 2: column orientation (M = j)
      if (tid == 0) {
        tc_fence_after();
        const uint32_t id128 = idesc_bf16(128, 128, 0, 0);
        for (int ks = 0; ks < p.N / 16; ++ks)
          mma_bf16(tT0, desc_c_kmajor(T, sB, ks), desc_c_kmajor(T, sC, ks), id128, ks > 0);
        for (int ks = 0; ks < 4; ++ks)
          mma_bf16(tT1, desc_tok_kmajor(sX, ks), desc_tok_kmajor(sY, ks), id128, ks > 0);
        mma_commit(&bar[1]);
      }
      if (!wait_mma(&bar[1], ph_mma)) ok = false;
      {  // column pass: thread owns token j; writes row j of A_hat = M^T
        const int j = J * kRows + tid;
        const bool cok = j < len;
        const float lj = cok ? lq[j] : 0.0f, dtj = cok ? dq[j] : 0.0f;
        const int sj = cok ? sq[j] : -3;
        float dd = 0.0f, dl = 0.0f;
        for (int q = 0; q < kRows / 16; ++q) {
          float cb[16], dm[16];
          tmem_ld16(tmem_addr(tT0, wlane, q * 16), cb);
          tmem_ld16(tmem_addr(tT1, wlane, q * 16), dm);
          uint32_t pk[8];
#pragma unroll
          for (int e = 0; e < 16; e += 2) {
            float mv[2];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
              const int i = I * kRows + q * 16 + e + u;
              float m = 0.0f;
              if (cok && j <= i && i < len && sq[i] == sj) {
                const float E = __expf(lq[i] - lj);
                const float cbE = cb[e + u] * E;
                m = cbE * dtj;
                dd += dm[e + u] * cbE;
                dl -= dm[e + u] * m;
              }
              mv[u] = m;
            }
            pk[e / 2] = pack2(mv[0], mv[1]);
          }
          uint8_t* blk = sA + (q / 4) * kTok;
          const uint32_t e0 = (q % 4) * 16;
          *reinterpret_cast<uint4*>(blk + swz128_off(tid, e0)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
          *reinterpret_cast<uint4*>(blk + swz128_off(tid, e0 + 8)) = make_uint4(pk[4], pk[5], pk[6], pk[7]);
        }
        if (cok) {
          dda[j] += dd;
          dla[j] += dl;
        }
      }
      fence_async_smem();
      tc_fence_before();
      __syncthreads();
      if (tid == 0) {  // dX_J += A_hat dY_I  (M = j, N = 64, K = tokens i)
        tc_fence_after();
        const uint32_t id64 = idesc_bf16(128, 64, 0, 1);
        for (int ks = 0; ks < kRows / 16; ++ks)
          mma_bf16(tDX, desc_tok_kmajor(sA, ks), desc_rows_mnmajor(sY, ks), id64, (!first || ks > 0));
        mma_commit(&bar[1]);
      }
      first = false;
      if (!wait_mma(&bar[1], ph_mma)) ok = false;
      if (diag) {  // epilogue of column block J (sX = x_J, sY = dy_J)
        const int j = J * kRows + tid;
        const bool cok = j < len;
        const float w = (cok && sq[j] == s_last) ? __expf(l_last - lq[j]) : 0.0f;
        const float u = w * (cok ? dq[j] : 0.0f);
        float du = 0.0f, dyx = 0.0f;
        __nv_bfloat16* dx = static_cast<__nv_bfloat16*>(f.dx);
        const long long xrow = (((long long)bi * p.L + t0 + j) * p.H + h) * 64;
        for (int q = 0; q < 4; ++q) {
          float a[16], s[16];
          tmem_ld16(tmem_addr(tDX, wlane, q * 16), a);
          tmem_ld16(tmem_addr(tDXS, wlane, q * 16), s);
          const uint4 x0 = *reinterpret_cast<const uint4*>(sX + swz128_off(tid, q * 16));
          const uint4 x1 = *reinterpret_cast<const uint4*>(sX + swz128_off(tid, q * 16 + 8));
          const uint4 y0 = *reinterpret_cast<const uint4*>(sY + swz128_off(tid, q * 16));
          const uint4 y1 = *reinterpret_cast<const uint4*>(sY + swz128_off(tid, q * 16 + 8));
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
          if (cok) {
            uint4* dst = reinterpret_cast<uint4*>(dx + xrow + q * 16);
            dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
            dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
          }
        }
        if (cok) {
          dda[j] += w * du;
          dla[j] -= u * du;
          udu_part += u * du;
          dD_part += dyx;
        }
        tc_fence_before();
        __syncthreads();
      }
    }
  }
  red[tid] = udu_part;
  red[kThr + tid] = dD_part;
  __syncthreads();
  for (int t = tid; t < len; t += kThr) {
    f.ddte[bh * p.Lp + t0 + t] = dda[t];
    f.dl[bh * p.Lp + t0 + t] = dla[t];
  }
  if (tid == 0) {
    float su = 0.0f, sd = 0.0f;
    for (int t = 0; t < kThr; ++t) {
      su += red[t];
      sd += red[kThr + t];
    }
    f.udu[bh * p.nc + c] = su;
    f.pdD[((long long)bi * p.nc + c) * p.H + h] = sd;
  }
  if (!ok) atomicOr(&f.hdr->status, kDevTimeout);
  tc_fence_before();
  __syncthreads();
  if (tid < 32) tmem_dealloc(tm, 512);
}

// ---------------------------------------------------------------------------
// Writes a row-scaled copy of a (128 x 64) token tile (row r scaled by s) into
// dst with the same swizzled layout (row r is owned by thread r).
__device__ __forceinline__ void scaled_copy(uint8_t* dst, const uint8_t* src, int r, float s) {
  for (int q = 0; q < 8; ++q) {
    const uint4 v = *reinterpret_cast<const uint4*>(src + swz128_off(r, q * 8));
    const uint32_t a[4] = {v.x, v.y, v.z, v.w};
    uint32_t o[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 x = unpack2(a[e]);
      o[e] = pack2(x.x * s, x.y * s);
    }
    *reinterpret_cast<uint4*>(dst + swz128_off(r, q * 8)) = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

__global__ void __launch_bounds__(kThr) chunk_bwd_dbc_tc_kernel(Plan p, Bufs f,
                                                                const __grid_constant__ CUtensorMap tmX,
                                                                const __grid_constant__ CUtensorMap tmY,
                                                                const __grid_constant__ CUtensorMap tmB,
                                                                const __grid_constant__ CUtensorMap tmC,
                                                                const __grid_constant__ CUtensorMap tmS,
                                                                const __grid_constant__ CUtensorMap tmH) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const Tiles T = tiles(p.N, p.Q);
  const int nb = (p.Q + kRows - 1) / kRows;
  uint8_t* sBT = sm;                  // own B block (group)
  uint8_t* sCT = sBT + T.cbytes;      // own C block (group)
  uint8_t* sXT = sCT + T.cbytes;      // own x block (head)
  uint8_t* sYT = sXT + kTok;          // own dy block (head)
  uint8_t* sS = sYT + kTok;           // dS (head)
  uint8_t* sH = sS + T.sbytes;        // H (head)
  uint8_t* sA = sH + T.sbytes;        // derived operand
  uint8_t* sP1 = sA + kAhat;          // partner B_J or C_I (only when nb > 1)
  uint8_t* sP2 = sP1 + (nb > 1 ? T.cbytes : 0);  // partner x_J or dy_I
  float* lq = reinterpret_cast<float*>(sP2 + (nb > 1 ? kTok : 0));
  float* dq = lq + p.Q;
  int* sq = reinterpret_cast<int*>(dq + p.Q);
  uint64_t* bar = reinterpret_cast<uint64_t*>(sq + p.Q);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + 2);

  const int TB = blockIdx.x % nb, c = blockIdx.x / nb;
  const int g = blockIdx.y, bi = blockIdx.z;
  const int tid = threadIdx.x, wlane = (tid >> 5) * 32;
  const int t0 = c * p.Q, len = min(p.Q, p.L - t0);
  const int own0 = TB * kRows;
  if (own0 >= len) return;  // uniform per CTA

  for (int t = tid; t < p.Q; t += kThr) sq[t] = t < len ? seg_of(p, f, bi, (long long)t0 + t) : -1;
  if (T.rows < kRows) {
    for (int idx = tid; idx < (kRows - T.rows) * 8; idx += kThr) {
      reinterpret_cast<uint4*>(sXT + T.rows * 128)[idx] = make_uint4(0, 0, 0, 0);
      reinterpret_cast<uint4*>(sYT + T.rows * 128)[idx] = make_uint4(0, 0, 0, 0);
    }
    // B and C are contracted over tokens here: their padding rows must be zero too
    const int per = (kRows - T.rows) * T.cw / 16;
    for (int idx = tid; idx < 2 * T.ncb * per; idx += kThr) {
      const int blk = idx / per, k = idx % per;
      uint8_t* base = (blk < T.ncb ? sBT : sCT) + (blk % T.ncb) * T.cblk + T.rows * T.cw;
      reinterpret_cast<uint4*>(base)[k] = make_uint4(0, 0, 0, 0);
    }
  }
  if (tid == 0) {
    mbar_init(&bar[0], 1);
    mbar_init(&bar[1], 1);
    mbar_fence_init();
  }
  if (tid < 32) tmem_alloc(tmem_slot, 512);
  fence_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tm = *tmem_slot;
  const uint32_t tDC = tm, tDB = tm + 128, tSC = tm + 256;
  const int s_in = seg_in_of(p, f, bi, c);
  const int s_last = seg_of(p, f, bi, (long long)t0 + len - 1);
  bool ok = true;
  uint32_t ph_ld = 0, ph_mma = 0;
  const uint32_t tok_bytes = (uint32_t)T.rows * 128u;
  const uint32_t c_bytes = (uint32_t)T.ncb * T.rows * T.cw;
  const uint32_t idN_kk = idesc_bf16(128, p.N, 0, 0);   // B operand K-major (H, dS)
  const uint32_t idN_kmn = idesc_bf16(128, p.N, 0, 1);  // B operand MN-major (B_J, C_I)
  const uint32_t id128 = idesc_bf16(128, 128, 0, 0);
  bool dc_started = false, db_started = false;

  if (tid == 0) {
    mbar_expect_tx(&bar[0], 2 * c_bytes);
    for (int q = 0; q < T.ncb; ++q) {
      tma_load_4d(sBT + q * T.cblk, &tmB, &bar[0], q * 64, g, t0 + own0, bi);
      tma_load_4d(sCT + q * T.cblk, &tmC, &bar[0], q * 64, g, t0 + own0, bi);
    }
  }
  if (!mbar_wait(&bar[0], ph_ld)) ok = false;
  ph_ld ^= 1;

  for (int hh = 0; hh < p.hpg; ++hh) {
    const int h = g * p.hpg + hh;
    const long long bh = (long long)bi * p.H + h;
    for (int t = tid; t < p.Q; t += kThr) {
      lq[t] = f.lcs[bh * p.Lp + t0 + t];
      dq[t] = f.dte[bh * p.Lp + t0 + t];
    }
    if (tid == 0) {
      mbar_expect_tx(&bar[0], 2 * tok_bytes + 2u * (uint32_t)p.N * 128u);
      tma_load_4d(sXT, &tmX, &bar[0], 0, h, t0 + own0, bi);
      tma_load_4d(sYT, &tmY, &bar[0], 0, h, t0 + own0, bi);
      tma_load_4d(sS, &tmS, &bar[0], 0, 0, c, (int)bh);
      tma_load_4d(sH, &tmH, &bar[0], 0, 0, c, (int)bh);
    }
    if (!mbar_wait(&bar[0], ph_ld)) ok = false;
    ph_ld ^= 1;
    __syncthreads();  // lq/dq of this head visible
    const int r = tid;
    // ---- dC rows (own block): partners J <= TB
    for (int J = 0; J <= TB; ++J) {
      const uint8_t* bJ = sBT;
      const uint8_t* xJ = sXT;
      tc_fence_before();
      fence_async_smem();  // shared reads of the tiles before the copies that overwrite them
      __syncthreads();  // all threads are past their previous barrier waits
      if (J != TB) {
        if (tid == 0) {
          mbar_expect_tx(&bar[0], tok_bytes + c_bytes);
          tma_load_4d(sP2, &tmX, &bar[0], 0, h, t0 + J * kRows, bi);
          for (int q = 0; q < T.ncb; ++q) tma_load_4d(sP1 + q * T.cblk, &tmB, &bar[0], q * 64, g, t0 + J * kRows, bi);
        }
        if (!mbar_wait(&bar[0], ph_ld)) ok = false;
        ph_ld ^= 1;
        bJ = sP1;
        xJ = sP2;
      }
      if (tid == 0) {  // dM = dy_T x_J^T  (M = i, N = j, K = 64)
        tc_fence_after();
        for (int ks = 0; ks < 4; ++ks)
          mma_bf16(tSC, desc_tok_kmajor(sYT, ks), desc_tok_kmajor(xJ, ks), id128, ks > 0);
        mma_commit(&bar[1]);
      }
      if (!wait_mma(&bar[1], ph_mma)) ok = false;
      {
        const int i = own0 + r;
        const bool rok = i < len;
        const float li = rok ? lq[i] : 0.0f;
        const int si = rok ? sq[i] : -2;
        for (int q = 0; q < kRows / 16; ++q) {
          float dm[16];
          tmem_ld16(tmem_addr(tSC, wlane, q * 16), dm);
          uint32_t pk[8];
#pragma unroll
          for (int e = 0; e < 16; e += 2) {
            float v[2];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
              const int j = J * kRows + q * 16 + e + u;
              v[u] = (rok && j <= i && sq[j] == si) ? dm[e + u] * __expf(li - lq[j]) * dq[j] : 0.0f;
            }
            pk[e / 2] = pack2(v[0], v[1]);
          }
          uint8_t* blk = sA + (q / 4) * kTok;
          const uint32_t e0 = (q % 4) * 16;
          *reinterpret_cast<uint4*>(blk + swz128_off(r, e0)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
          *reinterpret_cast<uint4*>(blk + swz128_off(r, e0 + 8)) = make_uint4(pk[4], pk[5], pk[6], pk[7]);
        }
      }
      fence_async_smem();
      tc_fence_before();
      __syncthreads();
      if (tid == 0) {  // dC_T += dCB B_J  (M = i, N = d_state, K = tokens j)
        tc_fence_after();
        for (int ks = 0; ks < kRows / 16; ++ks)
          mma_bf16(tDC, desc_tok_kmajor(sA, ks), desc_c_mnmajor(T, bJ, ks), idN_kmn, (dc_started || ks > 0));
        mma_commit(&bar[1]);
      }
      dc_started = true;
      if (!wait_mma(&bar[1], ph_mma)) ok = false;
    }
    // ---- carry: dC_T += diag(cv e^l) dy_T H   (M = i, N = d_state, K = 64)
    {
      const int i = own0 + r;
      const float s = (i < len && sq[i] == s_in) ? __expf(lq[i]) : 0.0f;
      scaled_copy(sA, sYT, r, s);
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    if (tid == 0) {
      tc_fence_after();
      for (int ks = 0; ks < 4; ++ks)
        mma_bf16(tDC, desc_tok_kmajor(sA, ks), desc_tok_kmajor(sH, ks), idN_kk, 1u);
      mma_commit(&bar[1]);
    }
    if (!wait_mma(&bar[1], ph_mma)) ok = false;
    // ---- dB cols (own block): partners I >= TB
    for (int I = nb - 1; I >= TB; --I) {
      if (I * kRows >= len) continue;
      const uint8_t* cI = sCT;
      const uint8_t* yI = sYT;
      tc_fence_before();
      fence_async_smem();  // shared reads of the tiles before the copies that overwrite them
      __syncthreads();  // all threads are past their previous barrier waits
      if (I != TB) {
        if (tid == 0) {
          mbar_expect_tx(&bar[0], tok_bytes + c_bytes);
          tma_load_4d(sP2, &tmY, &bar[0], 0, h, t0 + I * kRows, bi);
          for (int q = 0; q < T.ncb; ++q) tma_load_4d(sP1 + q * T.cblk, &tmC, &bar[0], q * 64, g, t0 + I * kRows, bi);
        }
        if (!mbar_wait(&bar[0], ph_ld)) ok = false;
        ph_ld ^= 1;
        cI = sP1;
        yI = sP2;
      }
      if (tid == 0) {  // dM^T = x_T dy_I^T  (M = j, N = i, K = 64)
        tc_fence_after();
        for (int ks = 0; ks < 4; ++ks)
          mma_bf16(tSC, desc_tok_kmajor(sXT, ks), desc_tok_kmajor(yI, ks), id128, ks > 0);
        mma_commit(&bar[1]);
      }
      if (!wait_mma(&bar[1], ph_mma)) ok = false;
      {
        const int j = own0 + r;
        const bool cok = j < len;
        const float lj = cok ? lq[j] : 0.0f, dtj = cok ? dq[j] : 0.0f;
        const int sj = cok ? sq[j] : -3;
        for (int q = 0; q < kRows / 16; ++q) {
          float dm[16];
          tmem_ld16(tmem_addr(tSC, wlane, q * 16), dm);
          uint32_t pk[8];
#pragma unroll
          for (int e = 0; e < 16; e += 2) {
            float v[2];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
              const int i = I * kRows + q * 16 + e + u;
              v[u] = (cok && j <= i && i < len && sq[i] == sj) ? dm[e + u] * __expf(lq[i] - lj) * dtj : 0.0f;
            }
            pk[e / 2] = pack2(v[0], v[1]);
          }
          uint8_t* blk = sA + (q / 4) * kTok;
          const uint32_t e0 = (q % 4) * 16;
          *reinterpret_cast<uint4*>(blk + swz128_off(r, e0)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
          *reinterpret_cast<uint4*>(blk + swz128_off(r, e0 + 8)) = make_uint4(pk[4], pk[5], pk[6], pk[7]);
        }
      }
      fence_async_smem();
      tc_fence_before();
      __syncthreads();
      if (tid == 0) {  // dB_T += dCB^T C_I  (M = j, N = d_state, K = tokens i)
        tc_fence_after();
        for (int ks = 0; ks < kRows / 16; ++ks)
          mma_bf16(tDB, desc_tok_kmajor(sA, ks), desc_c_mnmajor(T, cI, ks), idN_kmn, (db_started || ks > 0));
        mma_commit(&bar[1]);
      }
      db_started = true;
      if (!wait_mma(&bar[1], ph_mma)) ok = false;
    }
    // ---- state: dB_T += diag(u) x_T dS   (M = j, N = d_state, K = 64)
    {
      const int j = own0 + r;
      const bool cok = j < len;
      const float u = (cok && sq[j] == s_last) ? __expf(lq[len - 1] - lq[j]) * dq[j] : 0.0f;
      scaled_copy(sA, sXT, r, u);
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    if (tid == 0) {
      tc_fence_after();
      for (int ks = 0; ks < 4; ++ks)
        mma_bf16(tDB, desc_tok_kmajor(sA, ks), desc_tok_kmajor(sS, ks), idN_kk, 1u);
      mma_commit(&bar[1]);
    }
    if (!wait_mma(&bar[1], ph_mma)) ok = false;
    fence_async_smem();  // shared reads of the tiles before the copies that overwrite them
    __syncthreads();  // before the next head's loads overwrite x/dy/dS/H and lq/dq
  }
  // ---- epilogue: rows of dB and dC for the own block.  tcgen05.ld is a
  // warp-collective instruction: every lane executes it, only the stores are
  // guarded by the ragged end.
  {
    const int t = own0 + tid;
    const bool v = t < len;
    __nv_bfloat16* dB = static_cast<__nv_bfloat16*>(f.dB);
    __nv_bfloat16* dC = static_cast<__nv_bfloat16*>(f.dC);
    const long long row = (((long long)bi * p.L + t0 + t) * p.G + g) * p.N;
    for (int n0 = 0; n0 < p.N; n0 += 16) {
      float vb[16], vc[16];
      tmem_ld16(tmem_addr(tDB, wlane, n0), vb);
      tmem_ld16(tmem_addr(tDC, wlane, n0), vc);
      if (v) {
        uint4* ob = reinterpret_cast<uint4*>(dB + row + n0);
        uint4* oc = reinterpret_cast<uint4*>(dC + row + n0);
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

bool encode_all(const Plan& p, const Bufs& f, CUtensorMap* X, CUtensorMap* Y, CUtensorMap* B, CUtensorMap* C,
                CUtensorMap* S, CUtensorMap* H) {
  const Tiles T = tiles(p.N, p.Q);
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

bool chunk_bwd_pair_tc_supported(const Plan& p) {
  return p.dtype == SSD_BF16 && p.P == 64 && (p.Q == 64 || p.Q == 128 || p.Q == 256) &&
         (p.N == 16 || p.N == 32 || p.N == 64 || p.N == 128);
}

size_t chunk_bwd_pair_tc_smem(const Plan& p, bool dbc) {
  const Tiles T = tiles(p.N, p.Q);
  if (!dbc) {
    const bool alias = T.cbytes >= kAhat;
    size_t b = 2 * kTok + 2 * (size_t)T.cbytes + (alias ? 0 : kAhat) + 2 * (size_t)T.sbytes;
    return 1024 + b + 5 * p.Q * 4 + 3 * kThr * 4 + 64;
  }
  const int nb = (p.Q + kRows - 1) / kRows;
  size_t b = 2 * (size_t)T.cbytes + 2 * kTok + 2 * (size_t)T.sbytes + kAhat + (nb > 1 ? T.cbytes + kTok : 0);
  return 1024 + b + 3 * p.Q * 4 + 64;
}

cudaError_t launch_chunk_bwd_pair_tc(const Plan& p, const Bufs& f, cudaStream_t s) {
  CUtensorMap X, Y, B, C, S, H;
  if (!encode_all(p, f, &X, &Y, &B, &C, &S, &H)) return cudaErrorInvalidValue;
  set_kernel_name("chunk_bwd_tc");
  const size_t smem = chunk_bwd_pair_tc_smem(p, false);
  cudaError_t e = cudaFuncSetAttribute(chunk_bwd_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  chunk_bwd_tc_kernel<<<dim3(p.nc, p.H, p.b), kThr, smem, s>>>(p, f, X, Y, B, C, S, H);
  return cudaGetLastError();
}

cudaError_t launch_chunk_bwd_dbc_tc(const Plan& p, const Bufs& f, cudaStream_t s) {
  CUtensorMap X, Y, B, C, S, H;
  if (!encode_all(p, f, &X, &Y, &B, &C, &S, &H)) return cudaErrorInvalidValue;
  set_kernel_name("chunk_bwd_dbc_tc");
  const size_t smem = chunk_bwd_pair_tc_smem(p, true);
  cudaError_t e = cudaFuncSetAttribute(chunk_bwd_dbc_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const int nb = (p.Q + kRows - 1) / kRows;
  chunk_bwd_dbc_tc_kernel<<<dim3(p.nc * nb, p.G, p.b), kThr, smem, s>>>(p, f, X, Y, B, C, S, H);
  return cudaGetLastError();
}

}  // namespace ssd
