// k_chunk_simt.cu -- per-chunk kernels of the SSD layer on the CUDA cores
// (fp32 FMA with fp32 accumulation), for any supported dtype and shape.
//
// These are the fp32 path and the reference-shaped path for shapes the
// tensor-core kernels do not cover.  Notation (chunk c of row b, head h of
// group g, chunk-local token indices i, j < len):
//   l_i   chunk-local cumsum of dt_eff A_h (from the dt kernel)
//   E_ij  = exp(l_i - l_j) if j <= i and seg_i = seg_j, else 0
//   cv_i  = [seg_i = seg of token c*Q-1]   (token i sees the carry-in state)
//   sv_j  = [seg_j = seg of the chunk's last token]
//
//  chunk_state  S_c    = sum_j sv_j exp(l_last - l_j) dt_eff_j  x_j (outer) B_j
//  chunk_dstate dHloc  = sum_i cv_i exp(l_i) dy_i (outer) C_i
//  chunk_scan   y_i    = sum_j (C_i . B_j) E_ij dt_eff_j x_j + cv_i exp(l_i) H_in C_i + D_h x_i
//  chunk_bwd    every token gradient of the chunk (see chunk_bwd_simt)
//
// Page "llm-mamba-200" (gigipick.blogspot.com), section 3: carry-out state of
// a chunk passed as the carry-in of the next; section 4: parallel over the
// sequence (chunks) and over the state dimension.
#include "ssd_internal.cuh"

namespace ssd {

namespace {

constexpr int kThreads = 256;
constexpr int kJs = 32;  // tokens per staging step of chunk_state
constexpr int kTb = 32;  // token block of chunk_scan / chunk_bwd

template <typename T, bool kDstates>
__global__ void __launch_bounds__(kThreads) chunk_state_simt(Plan p, Bufs f) {
  extern __shared__ float smem[];
  const int c = blockIdx.x, h = blockIdx.y, bi = blockIdx.z;
  const int g = h / p.hpg;
  const int P = p.P, N = p.N;
  const int t0 = c * p.Q, len = min(p.Q, p.L - t0);
  const long long bh = (long long)bi * p.H + h;
  float* w = smem;            // Q weights
  float* Xs = w + p.Q;        // kJs x P
  float* Bs = Xs + kJs * P;   // kJs x N
  const float* lc = f.lcs + bh * p.Lp + t0;
  const float* de = f.dte + bh * p.Lp + t0;
  if (kDstates) {
    const int s_in = seg_in_of(p, f, bi, c);
    for (int j = threadIdx.x; j < p.Q; j += kThreads)
      w[j] = (j < len && seg_of(p, f, bi, (long long)t0 + j) == s_in) ? expf(lc[j]) : 0.0f;
  } else {
    const float l_last = lc[len - 1];
    const int s_last = seg_of(p, f, bi, (long long)t0 + len - 1);
    for (int j = threadIdx.x; j < p.Q; j += kThreads)
      w[j] = (j < len && seg_of(p, f, bi, (long long)t0 + j) == s_last)
                 ? expf(l_last - lc[j]) * de[j]
                 : 0.0f;
  }
  const T* Xg = static_cast<const T*>(kDstates ? f.dy : f.x);
  const T* Bg = static_cast<const T*>(kDstates ? f.C : f.B);
  constexpr int kMaxOut = 8192 / kThreads;
  const int nout = p.PN / kThreads;
  float acc[kMaxOut];
#pragma unroll
  for (int k = 0; k < kMaxOut; ++k) acc[k] = 0.0f;
  __syncthreads();
  for (int j0 = 0; j0 < len; j0 += kJs) {
    for (int idx = threadIdx.x; idx < kJs * P; idx += kThreads) {
      const int j = idx / P, pp = idx - j * P;
      float v = 0.0f;
      if (j0 + j < len) v = to_f(Xg[(((long long)bi * p.L + t0 + j0 + j) * p.H + h) * P + pp]) * w[j0 + j];
      Xs[idx] = v;
    }
    for (int idx = threadIdx.x; idx < kJs * N; idx += kThreads) {
      const int j = idx / N, n = idx - j * N;
      float v = 0.0f;
      if (j0 + j < len) v = to_f(Bg[(((long long)bi * p.L + t0 + j0 + j) * p.G + g) * N + n]);
      Bs[idx] = v;
    }
    __syncthreads();
#pragma unroll
    for (int k = 0; k < kMaxOut; ++k) {
      if (k < nout) {
        const int o = threadIdx.x + k * kThreads;  // o = n * P + p
        const int n = o / P, pp = o - n * P;
        float a = acc[k];
        for (int j = 0; j < kJs; ++j) a = fmaf(Xs[j * P + pp], Bs[j * N + n], a);
        acc[k] = a;
      }
    }
    __syncthreads();
  }
  float* out = (kDstates ? f.dHl : f.S) + (bh * p.nc + c) * p.PN;
#pragma unroll
  for (int k = 0; k < kMaxOut; ++k)
    if (k < nout) out[threadIdx.x + k * kThreads] = acc[k];
}

template <typename T>
__global__ void __launch_bounds__(kThreads) chunk_scan_simt(Plan p, Bufs f) {
  extern __shared__ float smem[];
  const int c = blockIdx.x, h = blockIdx.y, bi = blockIdx.z;
  const int g = h / p.hpg;
  const int P = p.P, N = p.N, N1 = N + 1;
  const int t0 = c * p.Q, len = min(p.Q, p.L - t0);
  const long long bh = (long long)bi * p.H + h;
  float* lq = smem;                                   // Q
  float* dq = lq + p.Q;                               // Q
  int* sq = reinterpret_cast<int*>(dq + p.Q);         // Q
  float* Hs = reinterpret_cast<float*>(sq + p.Q);     // P x (N+1)
  float* Cs = Hs + P * N1;                            // kTb x (N+1)
  float* Bs = Cs + kTb * N1;                          // kTb x (N+1)
  float* Xs = Bs + kTb * N1;                          // kTb x P
  float* Ms = Xs + kTb * P;                           // kTb x (kTb+1)
  const T* x = static_cast<const T*>(f.x);
  const T* Bg = static_cast<const T*>(f.B);
  const T* Cg = static_cast<const T*>(f.C);
  T* y = static_cast<T*>(f.y);
  for (int i = threadIdx.x; i < p.Q; i += kThreads) {
    lq[i] = f.lcs[bh * p.Lp + t0 + i];
    dq[i] = f.dte[bh * p.Lp + t0 + i];
    sq[i] = i < len ? seg_of(p, f, bi, (long long)t0 + i) : -1;
  }
  const T* hin = static_cast<const T*>(f.Hin) + (bh * p.nc + c) * p.PN;
  for (int idx = threadIdx.x; idx < p.PN; idx += kThreads) {
    const int n = idx / P, pp = idx - n * P;
    Hs[pp * N1 + n] = to_f(hin[idx]);
  }
  const int s_in = seg_in_of(p, f, bi, c);
  const float Dh = f.D[h];
  constexpr int kMaxY = kTb * 128 / kThreads;
  const int ny = kTb * P / kThreads;
  for (int i0 = 0; i0 < len; i0 += kTb) {
    for (int idx = threadIdx.x; idx < kTb * N; idx += kThreads) {
      const int i = idx / N, n = idx - i * N;
      Cs[i * N1 + n] = (i0 + i < len) ? to_f(Cg[(((long long)bi * p.L + t0 + i0 + i) * p.G + g) * N + n]) : 0.0f;
    }
    __syncthreads();
    float yacc[kMaxY];
#pragma unroll
    for (int k = 0; k < kMaxY; ++k) {
      yacc[k] = 0.0f;
      if (k < ny) {
        const int o = threadIdx.x + k * kThreads;
        const int i = o / P, pp = o - i * P;
        const int ii = i0 + i;
        if (ii < len && sq[ii] == s_in) {
          float s = 0.0f;
          for (int n = 0; n < N; ++n) s = fmaf(Cs[i * N1 + n], Hs[pp * N1 + n], s);
          yacc[k] = expf(lq[ii]) * s;
        }
      }
    }
    const int jend = min(i0 + kTb, len);
    for (int j0 = 0; j0 < jend; j0 += kTb) {
      for (int idx = threadIdx.x; idx < kTb * N; idx += kThreads) {
        const int j = idx / N, n = idx - j * N;
        Bs[j * N1 + n] = (j0 + j < len) ? to_f(Bg[(((long long)bi * p.L + t0 + j0 + j) * p.G + g) * N + n]) : 0.0f;
      }
      for (int idx = threadIdx.x; idx < kTb * P; idx += kThreads) {
        const int j = idx / P, pp = idx - j * P;
        Xs[idx] = (j0 + j < len) ? to_f(x[(((long long)bi * p.L + t0 + j0 + j) * p.H + h) * P + pp]) : 0.0f;
      }
      __syncthreads();
      for (int o = threadIdx.x; o < kTb * kTb; o += kThreads) {
        const int i = o / kTb, j = o - i * kTb;
        const int ii = i0 + i, jj = j0 + j;
        float v = 0.0f;
        if (jj <= ii && ii < len && sq[ii] == sq[jj]) {
          float s = 0.0f;
          for (int n = 0; n < N; ++n) s = fmaf(Cs[i * N1 + n], Bs[j * N1 + n], s);
          v = s * expf(lq[ii] - lq[jj]) * dq[jj];
        }
        Ms[i * (kTb + 1) + j] = v;
      }
      __syncthreads();
#pragma unroll
      for (int k = 0; k < kMaxY; ++k) {
        if (k < ny) {
          const int o = threadIdx.x + k * kThreads;
          const int i = o / P, pp = o - i * P;
          float a = yacc[k];
          for (int j = 0; j < kTb; ++j) a = fmaf(Ms[i * (kTb + 1) + j], Xs[j * P + pp], a);
          yacc[k] = a;
        }
      }
      __syncthreads();
    }
#pragma unroll
    for (int k = 0; k < kMaxY; ++k) {
      if (k < ny) {
        const int o = threadIdx.x + k * kThreads;
        const int i = o / P, pp = o - i * P;
        if (i0 + i < len) {
          const long long gi = (((long long)bi * p.L + t0 + i0 + i) * p.H + h) * P + pp;
          y[gi] = from_f<T>(yacc[k] + Dh * to_f(x[gi]));
        }
      }
    }
    __syncthreads();
  }
}

// Every token gradient of one chunk for one group: a CTA owns a block of kTb
// tokens of chunk c and walks the heads of the group in order, so that dB and
// dC (sums over the group's heads) are accumulated in one fixed order.
//   state part (dS = dL/dS_c, u_j = sv_j exp(l_last - l_j) dt_eff_j):
//     dx_j += u_j dS B_j;  dB_j += u_j dS^T x_j;  du_j = x_j^T dS B_j
//     ddt_eff_j += sv_j exp(l_last - l_j) du_j;  dl_j -= u_j du_j;  dl_last += sum_j u_j du_j
//   carry part (H = H_in[c]):  dC_i += cv_i e^{l_i} H^T dy_i;  dl_i += dy_i . (cv_i e^{l_i} H C_i)
//   intra part (M_ij = (C_i.B_j) E_ij dt_eff_j, dM_ij = dy_i . x_j):
//     dx_j += sum_i M_ij dy_i;  dC_i += sum_j dM_ij E_ij dt_eff_j B_j;
//     dB_j += sum_i dM_ij E_ij dt_eff_j C_i;  ddt_eff_j += sum_i dM_ij (C_i.B_j) E_ij;
//     dl_i += sum_j dM_ij M_ij;  dl_j -= sum_i dM_ij M_ij
//   skip part: dx_j += D_h dy_j;  dD_h += dy_j . x_j
// The dl_last term summed over the chunk goes to per-block partials folded by
// dt_bwd (the other dl_last term, a_c dL/da_c, comes from the reverse scan).
template <typename T>
__global__ void __launch_bounds__(kThreads) chunk_bwd_simt(Plan p, Bufs f) {
  extern __shared__ float smem[];
  const int tb = blockIdx.x, c = blockIdx.y;
  const int bi = blockIdx.z / p.G, g = blockIdx.z % p.G;
  const int P = p.P, N = p.N, N1 = N + 1, P1 = P + 1, T1 = kTb + 1;
  const int t0 = c * p.Q, len = min(p.Q, p.L - t0);
  const int o0 = tb * kTb;
  const int ntb = p.cb_ntb;
  if (o0 >= len) {  // a block past the ragged end: its partials are zero
    for (int hh = threadIdx.x; hh < p.hpg; hh += kThreads) {
      const int h = g * p.hpg + hh;
      const long long bh = (long long)bi * p.H + h;
      f.udu[(bh * p.nc + c) * ntb + tb] = 0.0f;
      f.pdD[(((long long)bi * p.nc + c) * ntb + tb) * p.H + h] = 0.0f;
    }
    return;
  }
  float* lq = smem;                                  // Q
  float* dq = lq + p.Q;                              // Q
  int* sq = reinterpret_cast<int*>(dq + p.Q);        // Q
  float* dSs = reinterpret_cast<float*>(sq + p.Q);   // P x (N+1)
  float* Hs = dSs + P * N1;                          // P x (N+1)
  float* Bt = Hs + P * N1;                           // kTb x (N+1) own B rows
  float* Ct = Bt + kTb * N1;                         // kTb x (N+1) own C rows
  float* Xt = Ct + kTb * N1;                         // kTb x (P+1) own x rows
  float* Yt = Xt + kTb * P1;                         // kTb x (P+1) own dy rows
  float* Bp = Yt + kTb * P1;                         // kTb x (N+1) partner B or C rows
  float* Xp = Bp + kTb * N1;                         // kTb x (P+1) partner x or dy rows (also scratch)
  float* M1 = Xp + kTb * P1;                         // 4 tiles kTb x (kTb+1)
  float* M2 = M1 + kTb * T1;
  float* M3 = M2 + kTb * T1;
  float* M4 = M3 + kTb * T1;
  float* dBa = M4 + kTb * T1;                        // kTb x N
  float* dCa = dBa + kTb * N;                        // kTb x N
  float* wv = dCa + kTb * N;                         // kTb
  float* uv = wv + kTb;                              // kTb
  float* cve = uv + kTb;                             // kTb
  float* duv = cve + kTb;                            // kTb
  float* dla = duv + kTb;                            // kTb
  float* dda = dla + kTb;                            // kTb
  float* red = dda + kTb;                            // kThreads

  const T* xg = static_cast<const T*>(f.x);
  const T* yg = static_cast<const T*>(f.dy);
  const T* Bg = static_cast<const T*>(f.B);
  const T* Cg = static_cast<const T*>(f.C);
  T* dxg = static_cast<T*>(f.dx);
  T* dBg = static_cast<T*>(f.dB);
  T* dCg = static_cast<T*>(f.dC);
  const int s_in = seg_in_of(p, f, bi, c);
  const int s_last = seg_of(p, f, bi, (long long)t0 + len - 1);
  const long long row0 = (long long)bi * p.L + t0;  // token index of the chunk start

  for (int i = threadIdx.x; i < p.Q; i += kThreads)
    sq[i] = i < len ? seg_of(p, f, bi, (long long)t0 + i) : -1;
  for (int idx = threadIdx.x; idx < kTb * N; idx += kThreads) {
    const int j = idx / N, n = idx - j * N;
    const bool ok = o0 + j < len;
    Bt[j * N1 + n] = ok ? to_f(Bg[((row0 + o0 + j) * p.G + g) * N + n]) : 0.0f;
    Ct[j * N1 + n] = ok ? to_f(Cg[((row0 + o0 + j) * p.G + g) * N + n]) : 0.0f;
    dBa[idx] = 0.0f;
    dCa[idx] = 0.0f;
  }
  constexpr int kMaxXP = kTb * 128 / kThreads;  // owned (j, p) pairs per thread
  const int nxp = kTb * P / kThreads;
  const int nxn = kTb * N / kThreads;

  for (int hh = 0; hh < p.hpg; ++hh) {
    const int h = g * p.hpg + hh;
    const long long bh = (long long)bi * p.H + h;
    __syncthreads();
    for (int i = threadIdx.x; i < p.Q; i += kThreads) {
      lq[i] = f.lcs[bh * p.Lp + t0 + i];
      dq[i] = f.dte[bh * p.Lp + t0 + i];
    }
    const T* dsg = static_cast<const T*>(f.dS) + (bh * p.nc + c) * p.PN;
    const T* hg = static_cast<const T*>(f.Hin) + (bh * p.nc + c) * p.PN;
    for (int idx = threadIdx.x; idx < p.PN; idx += kThreads) {
      const int n = idx / P, pp = idx - n * P;
      dSs[pp * N1 + n] = to_f(dsg[idx]);
      Hs[pp * N1 + n] = to_f(hg[idx]);
    }
    for (int idx = threadIdx.x; idx < kTb * P; idx += kThreads) {
      const int j = idx / P, pp = idx - j * P;
      const bool ok = o0 + j < len;
      Xt[j * P1 + pp] = ok ? to_f(xg[((row0 + o0 + j) * p.H + h) * P + pp]) : 0.0f;
      Yt[j * P1 + pp] = ok ? to_f(yg[((row0 + o0 + j) * p.H + h) * P + pp]) : 0.0f;
    }
    __syncthreads();
    if (threadIdx.x < kTb) {
      const int j = o0 + threadIdx.x;
      const bool ok = j < len;
      const float w = (ok && sq[j] == s_last) ? expf(lq[len - 1] - lq[j]) : 0.0f;
      wv[threadIdx.x] = w;
      uv[threadIdx.x] = w * (ok ? dq[j] : 0.0f);
      cve[threadIdx.x] = (ok && sq[j] == s_in) ? expf(lq[j]) : 0.0f;
      dla[threadIdx.x] = 0.0f;
      dda[threadIdx.x] = 0.0f;
    }
    __syncthreads();
    float dxa[kMaxXP];
    // (a) state part
#pragma unroll
    for (int k = 0; k < kMaxXP; ++k) {
      dxa[k] = 0.0f;
      if (k < nxp) {
        const int o = threadIdx.x + k * kThreads;
        const int j = o / P, pp = o - j * P;
        float s = 0.0f;
        for (int n = 0; n < N; ++n) s = fmaf(dSs[pp * N1 + n], Bt[j * N1 + n], s);
        dxa[k] = uv[j] * s;
        Xp[j * P1 + pp] = Xt[j * P1 + pp] * s;
      }
    }
    for (int k = 0; k < nxn; ++k) {
      const int o = threadIdx.x + k * kThreads;
      const int j = o / N, n = o - j * N;
      float s = 0.0f;
      for (int pp = 0; pp < P; ++pp) s = fmaf(Xt[j * P1 + pp], dSs[pp * N1 + n], s);
      dBa[o] = fmaf(uv[j], s, dBa[o]);
    }
    __syncthreads();
    if (threadIdx.x < kTb) {
      float du = 0.0f;
      for (int pp = 0; pp < P; ++pp) du += Xp[threadIdx.x * P1 + pp];
      duv[threadIdx.x] = du;
      dda[threadIdx.x] += wv[threadIdx.x] * du;
      dla[threadIdx.x] -= uv[threadIdx.x] * du;
    }
    __syncthreads();
    // (b) carry part
    for (int k = 0; k < nxp; ++k) {
      const int o = threadIdx.x + k * kThreads;
      const int i = o / P, pp = o - i * P;
      float s = 0.0f;
      for (int n = 0; n < N; ++n) s = fmaf(Hs[pp * N1 + n], Ct[i * N1 + n], s);
      Xp[i * P1 + pp] = Yt[i * P1 + pp] * s * cve[i];
    }
    for (int k = 0; k < nxn; ++k) {
      const int o = threadIdx.x + k * kThreads;
      const int i = o / N, n = o - i * N;
      float s = 0.0f;
      for (int pp = 0; pp < P; ++pp) s = fmaf(Yt[i * P1 + pp], Hs[pp * N1 + n], s);
      dCa[o] = fmaf(cve[i], s, dCa[o]);
    }
    __syncthreads();
    if (threadIdx.x < kTb) {
      float s = 0.0f;
      for (int pp = 0; pp < P; ++pp) s += Xp[threadIdx.x * P1 + pp];
      dla[threadIdx.x] += s;
    }
    __syncthreads();
    // (c) partners j <= i: own rows i get dC and dl
    for (int J = 0; J <= tb; ++J) {
      const int jp0 = J * kTb;
      for (int idx = threadIdx.x; idx < kTb * N; idx += kThreads) {
        const int j = idx / N, n = idx - j * N;
        Bp[j * N1 + n] = (jp0 + j < len) ? to_f(Bg[((row0 + jp0 + j) * p.G + g) * N + n]) : 0.0f;
      }
      for (int idx = threadIdx.x; idx < kTb * P; idx += kThreads) {
        const int j = idx / P, pp = idx - j * P;
        Xp[j * P1 + pp] = (jp0 + j < len) ? to_f(xg[((row0 + jp0 + j) * p.H + h) * P + pp]) : 0.0f;
      }
      __syncthreads();
      for (int o = threadIdx.x; o < kTb * kTb; o += kThreads) {
        const int i = o / kTb, j = o - i * kTb;
        const int ii = o0 + i, jj = jp0 + j;
        float v1 = 0.0f, v2 = 0.0f;
        if (jj <= ii && ii < len && sq[ii] == sq[jj]) {
          const float E = expf(lq[ii] - lq[jj]);
          float cb = 0.0f, dm = 0.0f;
          for (int n = 0; n < N; ++n) cb = fmaf(Ct[i * N1 + n], Bp[j * N1 + n], cb);
          for (int pp = 0; pp < P; ++pp) dm = fmaf(Yt[i * P1 + pp], Xp[j * P1 + pp], dm);
          const float Ed = E * dq[jj];
          v1 = dm * Ed;              // dCB_ij
          v2 = dm * (cb * Ed);       // dM_ij M_ij
        }
        M1[i * T1 + j] = v1;
        M2[i * T1 + j] = v2;
      }
      __syncthreads();
      for (int k = 0; k < nxn; ++k) {
        const int o = threadIdx.x + k * kThreads;
        const int i = o / N, n = o - i * N;
        float s = 0.0f;
        for (int j = 0; j < kTb; ++j) s = fmaf(M1[i * T1 + j], Bp[j * N1 + n], s);
        dCa[o] += s;
      }
      if (threadIdx.x < kTb) {
        float s = 0.0f;
        for (int j = 0; j < kTb; ++j) s += M2[threadIdx.x * T1 + j];
        dla[threadIdx.x] += s;
      }
      __syncthreads();
    }
    // (d) partners i >= j: own columns j get dx, dB, ddt_eff and dl
    for (int I = tb; I < ntb; ++I) {
      const int ip0 = I * kTb;
      if (ip0 >= len) break;
      for (int idx = threadIdx.x; idx < kTb * N; idx += kThreads) {
        const int i = idx / N, n = idx - i * N;
        Bp[i * N1 + n] = (ip0 + i < len) ? to_f(Cg[((row0 + ip0 + i) * p.G + g) * N + n]) : 0.0f;
      }
      for (int idx = threadIdx.x; idx < kTb * P; idx += kThreads) {
        const int i = idx / P, pp = idx - i * P;
        Xp[i * P1 + pp] = (ip0 + i < len) ? to_f(yg[((row0 + ip0 + i) * p.H + h) * P + pp]) : 0.0f;
      }
      __syncthreads();
      for (int o = threadIdx.x; o < kTb * kTb; o += kThreads) {
        const int i = o / kTb, j = o - i * kTb;
        const int ii = ip0 + i, jj = o0 + j;
        float v1 = 0.0f, v2 = 0.0f, v3 = 0.0f, v4 = 0.0f;
        if (jj <= ii && ii < len && sq[ii] == sq[jj]) {
          const float E = expf(lq[ii] - lq[jj]);
          float cb = 0.0f, dm = 0.0f;
          for (int n = 0; n < N; ++n) cb = fmaf(Bp[i * N1 + n], Bt[j * N1 + n], cb);
          for (int pp = 0; pp < P; ++pp) dm = fmaf(Xp[i * P1 + pp], Xt[j * P1 + pp], dm);
          const float Ed = E * dq[jj];
          v1 = cb * Ed;              // M_ij
          v2 = dm * Ed;              // dCB_ij
          v3 = dm * cb * E;          // d/d dt_eff_j
          v4 = dm * v1;              // dM_ij M_ij
        }
        M1[i * T1 + j] = v1;
        M2[i * T1 + j] = v2;
        M3[i * T1 + j] = v3;
        M4[i * T1 + j] = v4;
      }
      __syncthreads();
#pragma unroll
      for (int k = 0; k < kMaxXP; ++k) {
        if (k < nxp) {
          const int o = threadIdx.x + k * kThreads;
          const int j = o / P, pp = o - j * P;
          float s = dxa[k];
          for (int i = 0; i < kTb; ++i) s = fmaf(M1[i * T1 + j], Xp[i * P1 + pp], s);
          dxa[k] = s;
        }
      }
      for (int k = 0; k < nxn; ++k) {
        const int o = threadIdx.x + k * kThreads;
        const int j = o / N, n = o - j * N;
        float s = 0.0f;
        for (int i = 0; i < kTb; ++i) s = fmaf(M2[i * T1 + j], Bp[i * N1 + n], s);
        dBa[o] += s;
      }
      if (threadIdx.x < kTb) {
        float s3 = 0.0f, s4 = 0.0f;
        for (int i = 0; i < kTb; ++i) {
          s3 += M3[i * T1 + threadIdx.x];
          s4 += M4[i * T1 + threadIdx.x];
        }
        dda[threadIdx.x] += s3;
        dla[threadIdx.x] -= s4;
      }
      __syncthreads();
    }
    // (e) this head's outputs and partials
    const float Dh = f.D[h];
#pragma unroll
    for (int k = 0; k < kMaxXP; ++k) {
      if (k < nxp) {
        const int o = threadIdx.x + k * kThreads;
        const int j = o / P, pp = o - j * P;
        if (o0 + j < len)
          dxg[((row0 + o0 + j) * p.H + h) * P + pp] = from_f<T>(fmaf(Dh, Yt[j * P1 + pp], dxa[k]));
      }
    }
    if (threadIdx.x < kTb) {
      const int j = o0 + threadIdx.x;
      float r = 0.0f;
      if (j < len) {
        f.ddte[bh * p.Lp + t0 + j] = dda[threadIdx.x];
        f.dl[bh * p.Lp + t0 + j] = dla[threadIdx.x];
        for (int pp = 0; pp < P; ++pp) r = fmaf(Yt[threadIdx.x * P1 + pp], Xt[threadIdx.x * P1 + pp], r);
      }
      red[threadIdx.x] = r;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      float sd = 0.0f, su = 0.0f;
      for (int j = 0; j < kTb; ++j) {
        sd += red[j];
        su += uv[j] * duv[j];
      }
      f.pdD[(((long long)bi * p.nc + c) * ntb + tb) * p.H + h] = sd;
      f.udu[(bh * p.nc + c) * ntb + tb] = su;
    }
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < kTb * N; idx += kThreads) {
    const int j = idx / N, n = idx - j * N;
    if (o0 + j < len) {
      const long long gi = ((row0 + o0 + j) * p.G + g) * N + n;
      dBg[gi] = from_f<T>(dBa[idx]);
      dCg[gi] = from_f<T>(dCa[idx]);
    }
  }
}

size_t chunk_state_smem(const Plan& p) { return sizeof(float) * (p.Q + kJs * (p.P + p.N)); }
size_t chunk_scan_smem(const Plan& p) {
  return sizeof(float) * (3 * p.Q + p.P * (p.N + 1) + 2 * kTb * (p.N + 1) + kTb * p.P + kTb * (kTb + 1));
}
size_t chunk_bwd_smem(const Plan& p) {
  const size_t N1 = p.N + 1, P1 = p.P + 1;
  return sizeof(float) * (3 * p.Q + 2 * p.P * N1 + 3 * kTb * N1 + 3 * kTb * P1 + 4 * kTb * (kTb + 1) +
                          2 * kTb * p.N + 6 * kTb + kThreads);
}

template <typename K>
cudaError_t launch_with_smem(K kernel, dim3 grid, size_t smem, cudaStream_t s, const Plan& p,
                             const Bufs& f) {
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  kernel<<<grid, kThreads, smem, s>>>(p, f);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_chunk_state(const Plan& p, const Bufs& f, bool dstates, cudaStream_t s) {
  if (chunk_state_tc_supported(p)) return launch_chunk_state_tc(p, f, dstates, s);
  dim3 grid(p.nc, p.H, p.b);
  const size_t smem = chunk_state_smem(p);
  set_kernel_name(dstates ? "chunk_dstate_simt" : "chunk_state_simt");
  if (p.dtype == SSD_BF16)
    return dstates ? launch_with_smem(chunk_state_simt<__nv_bfloat16, true>, grid, smem, s, p, f)
                   : launch_with_smem(chunk_state_simt<__nv_bfloat16, false>, grid, smem, s, p, f);
  return dstates ? launch_with_smem(chunk_state_simt<float, true>, grid, smem, s, p, f)
                 : launch_with_smem(chunk_state_simt<float, false>, grid, smem, s, p, f);
}

cudaError_t launch_chunk_scan(const Plan& p, const Bufs& f, cudaStream_t s) {
  if (chunk_scan_tc_supported(p)) return launch_chunk_scan_tc(p, f, s);
  dim3 grid(p.nc, p.H, p.b);
  const size_t smem = chunk_scan_smem(p);
  set_kernel_name("chunk_scan_simt");
  if (p.dtype == SSD_BF16) return launch_with_smem(chunk_scan_simt<__nv_bfloat16>, grid, smem, s, p, f);
  return launch_with_smem(chunk_scan_simt<float>, grid, smem, s, p, f);
}

cudaError_t launch_chunk_bwd(const Plan& p, const Bufs& f, cudaStream_t s) {
  if (chunk_bwd_tc_supported(p)) return launch_chunk_bwd_tc(p, f, s);
  dim3 grid(p.cb_ntb, p.nc, p.b * p.G);
  const size_t smem = chunk_bwd_smem(p);
  set_kernel_name("chunk_bwd_simt");
  if (p.dtype == SSD_BF16) return launch_with_smem(chunk_bwd_simt<__nv_bfloat16>, grid, smem, s, p, f);
  return launch_with_smem(chunk_bwd_simt<float>, grid, smem, s, p, f);
}

size_t simt_max_smem(const Plan& p) {
  size_t a = chunk_state_smem(p), b = chunk_scan_smem(p), c = chunk_bwd_smem(p);
  return a > b ? (a > c ? a : c) : (b > c ? b : c);
}

}  // namespace ssd
