// ssd_api.cu -- the C ABI of libssd: argument validation, workspace planning
// and the launch sequences of the forward and backward passes.
#include <mutex>
#include <string.h>

#include "ssd_internal.cuh"

namespace ssd {

namespace {

constexpr int kMaxDevices = 64;
struct DevInfo {
  int cc_major = -1, cc_minor = -1, sms = 0;
};
DevInfo g_dev[kMaxDevices];
std::mutex g_dev_mu;

bool current_device_info(DevInfo* out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return false;
  std::lock_guard<std::mutex> lk(g_dev_mu);
  DevInfo& d = g_dev[dev];
  if (d.cc_major < 0) {
    if (cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      d.cc_major = -1;
      return false;
    }
  }
  *out = d;
  return true;
}

bool pow2_in(int64_t v, int64_t lo, int64_t hi) {
  return v >= lo && v <= hi && (v & (v - 1)) == 0;
}

size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

// Validates the problem and fills the plan; returns SSD_OK or an error code.
int make_plan(const ssd_problem* pr, Plan* p) {
  if (!pr) return SSD_ERR_INVALID_ARGUMENT;
  if (pr->batch < 1 || pr->seqlen < 1 || pr->nheads < 1 || pr->headdim < 1 || pr->dstate < 1 ||
      pr->ngroups < 1 || pr->chunk_size < 1)
    return SSD_ERR_INVALID_ARGUMENT;
  if (pr->nheads % pr->ngroups != 0) return SSD_ERR_INVALID_ARGUMENT;
  if (pr->dtype != SSD_F32 && pr->dtype != SSD_BF16) return SSD_ERR_INVALID_ARGUMENT;
  if (pr->flags & ~(SSD_HAS_INIT | SSD_HAS_SEQ_IDX | SSD_HAS_DFINAL | SSD_WANT_DINIT | SSD_KEEP_FWD_STATES |
                    SSD_TEST_DROP_SCAN_PUBLISH | SSD_PATH_MULTI_KERNEL | SSD_PATH_SINGLE_PASS |
                    SSD_TEST_FEW_CTAS | SSD_SCAN_WARP_SHUFFLE))
    return SSD_ERR_INVALID_ARGUMENT;
  if (pr->chunk_size > 256 || pr->chunk_size % 16 != 0) return SSD_ERR_UNSUPPORTED;
  if (!pow2_in(pr->headdim, 16, 128) || !pow2_in(pr->dstate, 16, 128)) return SSD_ERR_UNSUPPORTED;
  if (pr->headdim * pr->dstate > 8192) return SSD_ERR_UNSUPPORTED;
  // 32-bit grid dimensions and 2^31 elements per tensor
  const int64_t nc = (pr->seqlen + pr->chunk_size - 1) / pr->chunk_size;
  if (pr->batch > 65535 || pr->nheads > 65535 || nc > (1 << 30)) return SSD_ERR_UNSUPPORTED;
  const int64_t big = pr->batch * (nc * pr->chunk_size) * pr->nheads *
                      (pr->headdim > pr->dstate ? pr->headdim : pr->dstate);
  if (big >= (int64_t(1) << 40)) return SSD_ERR_UNSUPPORTED;

  p->b = (int)pr->batch;
  p->L = (int)pr->seqlen;
  p->H = (int)pr->nheads;
  p->P = (int)pr->headdim;
  p->N = (int)pr->dstate;
  p->G = (int)pr->ngroups;
  // The chunk length is a blocking choice: the chunked evaluation gives the
  // result of the recurrence for any chunk length (up to rounding).  The
  // tensor-core path (bf16, headdim 64, d_state 16..128, at most 256 heads
  // per group) evaluates chunks of 128 tokens, its MMA tile, whatever
  // chunk_size asks; the CUDA-core path uses chunk_size as given.
  const bool tc_path = pr->dtype == SSD_BF16 && pr->headdim == 64 && pr->dstate >= 16 &&
                       pr->nheads / pr->ngroups <= 256;
  p->Q = tc_path ? 128 : (int)pr->chunk_size;
  p->nc = (p->L + p->Q - 1) / p->Q;
  p->PN = p->P * p->N;
  p->hpg = p->H / p->G;
  p->dtype = pr->dtype;
  p->flags = pr->flags;
  {
    // FNV-1a over the shape, the evaluation chunk and the inputs' presence
    uint32_t hsh = 2166136261u;
    const int64_t keys[] = {pr->batch, pr->seqlen, pr->nheads, pr->headdim, pr->dstate, pr->ngroups,
                            (int64_t)p->Q, (int64_t)pr->dtype,
                            (int64_t)(pr->flags & (SSD_HAS_INIT | SSD_HAS_SEQ_IDX))};
    for (int64_t k : keys)
      for (int byte = 0; byte < 8; ++byte) hsh = (hsh ^ (uint32_t)((k >> (8 * byte)) & 0xff)) * 16777619u;
    hsh &= ~(uint32_t)kKeptF32;  // bit 0 tells which forward kept the intermediates
    p->kept_sig = (int)(hsh == 0 ? 2u : hsh);
    p->kept_mode = 0;
    p->kept_sig_write = 0;
  }
  p->Lp = (long long)p->nc * p->Q;
  p->sp_neblk = (p->PN + kSpElems - 1) / kSpElems;
  p->sp_nseg = (p->nc + kSpSegF - 1) / kSpSegF;
  p->sp_nseg_b = (p->nc + kSpSegB - 1) / kSpSegB;
  p->sp_nslot = p->sp_nseg > p->sp_nseg_b ? p->sp_nseg : p->sp_nseg_b;
  p->sp_chains = p->b * p->H * p->sp_neblk;
  // per-chunk partial slots of the chunk-backward kernel: one per chunk on
  // the tensor-core path, one per 32-token block on the CUDA-core path
  // per-chunk partial slots of the chunk-backward kernel: one per warp row
  // block on the tensor-core path, one per 32-token block on the CUDA-core path
  p->cb_ntb = chunk_bwd_tc_supported(*p) ? 4 : (p->Q + 31) / 32;
  p->da_stride = p->sp_neblk > 16 ? p->sp_neblk : 16;
  p->da_nsum = p->sp_neblk;

  const size_t f4 = sizeof(float);
  const size_t bh = (size_t)p->b * p->H;
  const size_t states = bh * p->nc * p->PN * f4;
  size_t off = sizeof(WsHeader);
  auto take = [&](size_t bytes) {
    size_t o = off;
    off = align256(off + bytes);
    return o;
  };
  p->off_dte = take(bh * p->Lp * f4);
  p->off_lcs = take(bh * p->Lp * f4);
  p->off_achunk = take(bh * p->nc * f4);
  p->off_S = take(states);
  p->off_Hin = take(states / 4 * (p->dtype == SSD_BF16 ? 2 : 4));
  const size_t lb = (size_t)p->sp_chains * p->sp_nslot;
  p->off_agg = take(lb * kSpElems * f4);
  p->off_incl = take(lb * kSpElems * f4);
  p->off_flags_fwd = take(lb * sizeof(int));
  p->off_flags_bwd = take(lb * sizeof(int));
  p->fwd_bytes = off;
  p->off_dS = take(states / 4 * (p->dtype == SSD_BF16 ? 2 : 4));
  p->off_dHl = take(states);
  p->off_dapart = take(bh * p->nc * p->da_stride * f4);
  p->off_dl = take(bh * p->Lp * f4);
  p->off_ddte = take(bh * p->Lp * f4);
  p->off_udu = take(bh * p->nc * p->cb_ntb * f4);
  p->off_pdA = take(bh * p->nc * f4);
  p->off_pdb = take(bh * p->nc * f4);
  p->off_pdD = take(bh * p->nc * p->cb_ntb * f4);
  p->bwd_bytes = off;
  return SSD_OK;
}

bool misaligned(const void* ptr) { return ptr && (reinterpret_cast<uintptr_t>(ptr) & 15u); }

void bind_workspace(const Plan& p, void* ws, bool bwd, Bufs* f) {
  char* w = static_cast<char*>(ws);
  f->hdr = reinterpret_cast<WsHeader*>(w);
  f->dte = reinterpret_cast<float*>(w + p.off_dte);
  f->lcs = reinterpret_cast<float*>(w + p.off_lcs);
  f->achunk = reinterpret_cast<float*>(w + p.off_achunk);
  f->S = reinterpret_cast<float*>(w + p.off_S);
  f->Hin = w + p.off_Hin;
  f->agg = reinterpret_cast<float*>(w + p.off_agg);
  f->incl = reinterpret_cast<float*>(w + p.off_incl);
  f->flags_fwd = reinterpret_cast<int*>(w + p.off_flags_fwd);
  f->flags_bwd = reinterpret_cast<int*>(w + p.off_flags_bwd);
  if (bwd) {
    f->dS = w + p.off_dS;
    f->dl = reinterpret_cast<float*>(w + p.off_dl);
    f->ddte = reinterpret_cast<float*>(w + p.off_ddte);
    f->udu = reinterpret_cast<float*>(w + p.off_udu);
    f->dHl = reinterpret_cast<float*>(w + p.off_dHl);
    f->dapart = reinterpret_cast<float*>(w + p.off_dapart);
    f->pdA = reinterpret_cast<float*>(w + p.off_pdA);
    f->pdb = reinterpret_cast<float*>(w + p.off_pdb);
    f->pdD = reinterpret_cast<float*>(w + p.off_pdD);
  }
}

int check_device() {
  DevInfo d;
  if (!current_device_info(&d)) return SSD_ERR_CUDA;
  if (d.cc_major != 10 || d.cc_minor != 3) return SSD_ERR_UNSUPPORTED;
  return SSD_OK;
}

// The single-pass forward runs one CTA per (batch row, head) chain and walks
// its chunks in order: it is chosen where the shape is in its set and there
// are chains enough to fill most of the GPU.
bool enough_chains(const Plan& p) {
  if (p.flags & SSD_PATH_SINGLE_PASS) return true;
  return (long long)p.b * p.H * 4 >= (long long)device_sm_count() * 3;
}
bool use_fused_fwd(const Plan& p) {
  if (p.flags & (SSD_PATH_MULTI_KERNEL | SSD_TEST_DROP_SCAN_PUBLISH)) return false;
  return ssd_fwd_fused_supported(p) && enough_chains(p);
}
bool use_state_chains(const Plan& p) {
  if (p.flags & (SSD_PATH_MULTI_KERNEL | SSD_TEST_DROP_SCAN_PUBLISH)) return false;
  return state_chain_supported(p) && enough_chains(p);
}

#define SSD_LAUNCH(expr)                        \
  do {                                          \
    prof_before(s);                             \
    cudaError_t e_ = (expr);                    \
    prof_after(s);                              \
    if (e_ != cudaSuccess) return SSD_ERR_CUDA; \
  } while (0)

}  // namespace

int device_sm_count() {
  DevInfo d;
  return current_device_info(&d) ? d.sms : 148;
}

int device_check() { return check_device(); }

}  // namespace ssd

using namespace ssd;

extern "C" {

size_t ssd_fwd_workspace_bytes(const ssd_problem* prob) {
  Plan p;
  return make_plan(prob, &p) == SSD_OK ? p.fwd_bytes : 0;
}

size_t ssd_bwd_workspace_bytes(const ssd_problem* prob) {
  Plan p;
  return make_plan(prob, &p) == SSD_OK ? p.bwd_bytes : 0;
}

int ssd_fwd(const ssd_problem* prob, const void* x, const void* dt, const float* dt_bias,
            const float* A, const void* B, const void* C, const float* D,
            const float* initial_states, const int32_t* seq_idx, void* y, float* final_states,
            void* workspace, size_t workspace_bytes, ssd_stream_t stream) {
  Plan p;
  int rc = make_plan(prob, &p);
  if (rc != SSD_OK) return rc;
  if (p.flags & (SSD_HAS_DFINAL | SSD_WANT_DINIT)) return SSD_ERR_INVALID_ARGUMENT;
  if (!x || !dt || !dt_bias || !A || !B || !C || !D || !y || !workspace)
    return SSD_ERR_INVALID_ARGUMENT;
  if (((p.flags & SSD_HAS_INIT) != 0) != (initial_states != nullptr)) return SSD_ERR_INVALID_ARGUMENT;
  if (((p.flags & SSD_HAS_SEQ_IDX) != 0) != (seq_idx != nullptr)) return SSD_ERR_INVALID_ARGUMENT;
  const void* ptrs[] = {x, dt, dt_bias, A, B, C, D, initial_states, seq_idx, y, final_states, workspace};
  for (const void* q : ptrs)
    if (misaligned(q)) return SSD_ERR_INVALID_ARGUMENT;
  if (workspace_bytes < p.fwd_bytes) return SSD_ERR_WORKSPACE_TOO_SMALL;
  rc = check_device();
  if (rc != SSD_OK) return rc;

  Bufs f;
  memset(&f, 0, sizeof(f));
  f.x = x; f.dt = dt; f.dt_bias = dt_bias; f.A = A; f.B = B; f.C = C; f.D = D;
  f.init = initial_states; f.seq = seq_idx; f.y = y; f.final_states = final_states;
  bind_workspace(p, workspace, false, &f);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // every forward writes the kept-intermediates stamp: this problem's
  // signature if it keeps them (both paths leave them in the workspace; the
  // separate kernels' scan also keeps the fp32 carry-in states), else none
  const bool keep = (p.flags & SSD_KEEP_FWD_STATES) != 0;
  const bool fused = use_fused_fwd(p);
  p.kept_mode = 1;
  p.kept_sig_write = keep ? (p.kept_sig | (fused ? 0 : kKeptF32)) : 0;
  if (fused) {
    // no scan flags or tickets to reset, only the status word
    SSD_LAUNCH(launch_status_reset(p, f, s));
    SSD_LAUNCH(launch_ssd_fwd_fused(p, f, s));
    return SSD_OK;
  }
  SSD_LAUNCH(launch_dt_cumsum(p, f, s));
  SSD_LAUNCH(launch_chunk_state(p, f, false, s));
  SSD_LAUNCH(launch_state_passing(p, f, false, keep, s));
  SSD_LAUNCH(launch_chunk_scan(p, f, s));
  return SSD_OK;
}

int ssd_bwd(const ssd_problem* prob, const void* x, const void* dt, const float* dt_bias,
            const float* A, const void* B, const void* C, const float* D,
            const float* initial_states, const int32_t* seq_idx, const void* dy,
            const float* dfinal_states, void* dx, void* ddt, float* ddt_bias, float* dA,
            void* dB, void* dC, float* dD, float* dinitial_states, void* workspace,
            size_t workspace_bytes, ssd_stream_t stream) {
  Plan p;
  int rc = make_plan(prob, &p);
  if (rc != SSD_OK) return rc;
  if (!x || !dt || !dt_bias || !A || !B || !C || !D || !dy || !dx || !ddt || !ddt_bias || !dA ||
      !dB || !dC || !dD || !workspace)
    return SSD_ERR_INVALID_ARGUMENT;
  if (((p.flags & SSD_HAS_INIT) != 0) != (initial_states != nullptr)) return SSD_ERR_INVALID_ARGUMENT;
  if (((p.flags & SSD_HAS_SEQ_IDX) != 0) != (seq_idx != nullptr)) return SSD_ERR_INVALID_ARGUMENT;
  if (((p.flags & SSD_HAS_DFINAL) != 0) != (dfinal_states != nullptr)) return SSD_ERR_INVALID_ARGUMENT;
  if (((p.flags & SSD_WANT_DINIT) != 0) != (dinitial_states != nullptr)) return SSD_ERR_INVALID_ARGUMENT;
  const void* ptrs[] = {x, dt, dt_bias, A, B, C, D, initial_states, seq_idx, dy, dfinal_states,
                        dx, ddt, ddt_bias, dA, dB, dC, dD, dinitial_states, workspace};
  for (const void* q : ptrs)
    if (misaligned(q)) return SSD_ERR_INVALID_ARGUMENT;
  if (workspace_bytes < p.bwd_bytes) return SSD_ERR_WORKSPACE_TOO_SMALL;
  rc = check_device();
  if (rc != SSD_OK) return rc;

  Bufs f;
  memset(&f, 0, sizeof(f));
  f.x = x; f.dt = dt; f.dt_bias = dt_bias; f.A = A; f.B = B; f.C = C; f.D = D;
  f.init = initial_states; f.seq = seq_idx; f.dy = dy; f.dfinal = dfinal_states;
  f.dx = dx; f.ddt = ddt; f.ddt_bias = ddt_bias; f.dA = dA; f.dB = dB; f.dC = dC; f.dD = dD;
  f.dinit = dinitial_states;
  f.final_states = nullptr;  // the recomputed forward does not write final_states
  bind_workspace(p, workspace, true, &f);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (use_state_chains(p)) {
    // one pass per chain, forward then reverse (16 dL/da_c slots per chunk)
    p.da_nsum = 16;
    if (p.flags & SSD_KEEP_FWD_STATES) {
      // dt_eff, the chunk cumsums and decays and the carry-in states are the
      // forward's: check the stamp (in the status word) instead of recomputing
      p.kept_mode = 2;
      SSD_LAUNCH(launch_status_reset(p, f, s));
    } else {
      SSD_LAUNCH(launch_dt_cumsum(p, f, s));
      SSD_LAUNCH(launch_state_chain(p, f, false, s));
    }
    SSD_LAUNCH(launch_state_chain(p, f, true, s));
  } else {
    if ((p.flags & SSD_KEEP_FWD_STATES) && !use_fused_fwd(p)) {
      // dt_eff, the chunk cumsums and decays and the carry-in states, bf16
      // and fp32, are the separate-kernel forward's: check the stamp
      p.kept_mode = 3;
      SSD_LAUNCH(launch_kept_scan_reset(p, f, s));
    } else {
      // recompute the forward intermediates: dt_eff, chunk cumsums, carry-in states
      SSD_LAUNCH(launch_dt_cumsum(p, f, s));
      SSD_LAUNCH(launch_chunk_state(p, f, false, s));
      SSD_LAUNCH(launch_state_passing(p, f, false, true, s));
    }
    // gradient of the carry-in states from y, then the reverse state-passing scan
    SSD_LAUNCH(launch_chunk_state(p, f, true, s));
    SSD_LAUNCH(launch_state_passing(p, f, true, false, s));
  }
  SSD_LAUNCH(launch_chunk_bwd(p, f, s));
  // the tensor-core dB/dC kernel also forms ddt and the dA, ddt_bias partials
  if (!chunk_bwd_tc_supported(p)) SSD_LAUNCH(launch_dt_bwd(p, f, s));
  SSD_LAUNCH(launch_param_reduce(p, f, s));
  return SSD_OK;
}

const char* ssd_status_string(int status) {
  switch (status) {
    case SSD_OK: return "ok";
    case SSD_ERR_INVALID_ARGUMENT: return "invalid argument";
    case SSD_ERR_UNSUPPORTED: return "unsupported problem or device";
    case SSD_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case SSD_ERR_CUDA: return "CUDA error";
    case SSD_ERR_TIMEOUT: return "device-side wait timed out";
    case SSD_ERR_NO_KEPT_STATES: return "no kept forward intermediates of this problem in the workspace";
    default: return "unknown status";
  }
}

int ssd_read_device_status(const void* workspace, ssd_stream_t stream) {
  if (!workspace) return SSD_ERR_INVALID_ARGUMENT;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int st = 0;
  if (cudaMemcpyAsync(&st, workspace, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return SSD_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return SSD_ERR_CUDA;
  if (st & kDevTimeout) return SSD_ERR_TIMEOUT;
  return (st & kDevNoKept) ? SSD_ERR_NO_KEPT_STATES : SSD_OK;
}

const char* ssd_version(void) { return "libssd 0.1 sm_103a"; }

}  // extern "C"
