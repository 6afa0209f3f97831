// ssd_internal.cuh -- plan of one SSD problem (dimensions, workspace carve-up,
// kernel tiling) shared by the host entry points and the kernels of libssd.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "ssd.h"  // include/ (on the include path)

namespace ssd {

// Status bits the kernels OR into the device status word.
enum : int { kDevTimeout = 1, kDevNoKept = 2 };

// Bit 0 of the kept-intermediates stamp: the forward that wrote it also kept
// the fp32 carry-in states (the separate-kernel forward, whose scan writes
// them over the chunk states).  The rest of the stamp is the problem's
// signature, whose bit 0 is always clear.
constexpr int kKeptF32 = 1;

// State-passing scan tiling: one CTA scans kSpElems consecutive state elements
// (kSpThreads threads x 4 floats) over a segment of consecutive chunks:
// kSpSegF in the forward scan, kSpSegB in the reverse scan (which also stages
// the fp32 carry-in states, so its segments are half as long).
constexpr int kSpThreads = 128;
constexpr int kSpElems = kSpThreads * 4;
constexpr int kSpSegF = 16;
constexpr int kSpSegB = 8;

// Workspace header (first 256 bytes): device status word, then the tile
// tickets of the forward and backward state-passing scans.
struct WsHeader {
  int status;
  int ticket_fwd;
  int ticket_bwd;
  int kept_sig;  // signature of the problem whose forward intermediates the workspace holds, or 0
  int pad[60];
};
static_assert(sizeof(WsHeader) == 256, "header size");

struct Plan {
  // dimensions
  int b, L, H, P, N, G, Q, nc, PN, hpg;  // hpg = heads per group
  int dtype, flags;
  // nonzero signature of the problem's shape (the kept-intermediates stamp;
  // bit 0 clear) and what the launch that resets the status word does with
  // the stamp: 0 leave it, 1 write kept_sig_write, 2 check it against
  // kept_sig whatever its kKeptF32 bit, 3 check it against kept_sig with
  // the kKeptF32 bit set
  int kept_sig, kept_mode, kept_sig_write;
  long long Lp;                          // nc * Q (padded tokens per row)
  // state-passing scan tiling
  int sp_neblk, sp_nseg, sp_nseg_b, sp_nslot, sp_chains;  // chains = b * H * neblk; nslot = max segments
  // chunk-backward token blocks per chunk
  int cb_ntb;
  // dL/da_c partial slots per chunk: da_stride allocated (at least 16),
  // da_nsum written by the launch that forms them and summed in that order
  int da_stride, da_nsum;
  // workspace offsets in bytes (0 = absent)
  size_t off_dte, off_lcs, off_achunk;   // (b,H,Lp) f32, (b,H,Lp) f32, (b,H,nc) f32
  // Chunk-state tensors are stored (b, H, nc, N, P): for each state index n a
  // row of headdim values (the public initial/final states are (b, H, P, N)).
  size_t off_S;                          // (b,H,nc,N,P) f32: chunk states; in the backward,
                                         // then the fp32 carry-in states (in place)
  size_t off_Hin;                        // (b,H,nc,N,P) dtype: carry-in states
  size_t off_agg, off_incl;              // (chains, nslot, kSpElems) f32 each
  size_t off_flags_fwd, off_flags_bwd;   // (chains, nslot) int32 each
  // backward only
  size_t off_dS;                         // (b,H,nc,N,P) dtype: dL/dS_c
  size_t off_dHl;                        // (b,H,nc,N,P) f32: dL/dH_in[c] from the chunk outputs
  size_t off_dapart;                     // (b,H,nc,da_stride) f32: partial sums of dL/da_c
  size_t off_dl, off_ddte;               // (b,H,Lp) f32 each
  size_t off_udu;                        // (b,H,nc,cb_ntb) f32
  size_t off_pdA, off_pdb;               // (b,nc,H) f32 partials of dA, ddt_bias
  size_t off_pdD;                        // (b,nc,cb_ntb,H) f32 partials of dD
  size_t fwd_bytes, bwd_bytes;
};

// Device pointers of one call, passed by value to every kernel.
struct Bufs {
  const void* x;
  const void* dt;
  const float* dt_bias;
  const float* A;
  const void* B;
  const void* C;
  const float* D;
  const float* init;
  const int32_t* seq;
  void* y;
  float* final_states;
  // backward
  void* dS;  // storage dtype of the problem
  const void* dy;
  const float* dfinal;
  void* dx;
  void* ddt;
  float* ddt_bias;
  float* dA;
  void* dB;
  void* dC;
  float* dD;
  float* dinit;
  // workspace views
  WsHeader* hdr;
  float* dte;
  float* lcs;
  float* achunk;
  float* S;
  void* Hin;  // storage dtype of the problem
  float* agg;
  float* incl;
  int* flags_fwd;
  int* flags_bwd;
  float* dl;
  float* ddte;
  float* udu;
  float* dHl;
  float* dapart;
  float* pdA;
  float* pdb;
  float* pdD;
};

// Loads/stores of the storage dtype as fp32.
__device__ __forceinline__ float to_f(float v) { return v; }
__device__ __forceinline__ float to_f(__nv_bfloat16 v) { return __bfloat162float(v); }
template <typename T>
__device__ __forceinline__ T from_f(float v);
template <>
__device__ __forceinline__ float from_f<float>(float v) { return v; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float v) {
  return __float2bfloat16_rn(v);
}

// Segment id of token t of row bi (0 when there is no seq_idx).
__device__ __forceinline__ int seg_of(const Plan& p, const Bufs& f, int bi, long long t) {
  return (f.seq != nullptr) ? __ldg(f.seq + (long long)bi * p.L + t) : 0;
}
// Segment id live at the end of the previous chunk (token c*Q - 1; the first
// chunk takes the id of token 0, so the initial state reaches segment 0).
__device__ __forceinline__ int seg_in_of(const Plan& p, const Bufs& f, int bi, int c) {
  long long t = (long long)c * p.Q - 1;
  return seg_of(p, f, bi, t < 0 ? 0 : t);
}

// Host launchers (each returns the launch's cudaError_t).
cudaError_t launch_dt_cumsum(const Plan& p, const Bufs& f, cudaStream_t s);
cudaError_t launch_status_reset(const Plan& p, const Bufs& f, cudaStream_t s);
// The reset of a backward that runs the reverse scan without the forward's
// recompute (which otherwise does it): zero the reverse scan's flags and
// ticket, clear the status word and check the stamp (kept_mode 3).
cudaError_t launch_kept_scan_reset(const Plan& p, const Bufs& f, cudaStream_t s);
// backward: the reverse scan (dS, dinit, dL/da_c partials); keep_f32 (forward
// only): also keep the fp32 carry-in states, in place over the chunk states.
cudaError_t launch_state_passing(const Plan& p, const Bufs& f, bool backward, bool keep_f32, cudaStream_t s);
cudaError_t launch_chunk_state(const Plan& p, const Bufs& f, bool dstates, cudaStream_t s);
cudaError_t launch_chunk_scan(const Plan& p, const Bufs& f, cudaStream_t s);
cudaError_t launch_chunk_bwd(const Plan& p, const Bufs& f, cudaStream_t s);
cudaError_t launch_dt_bwd(const Plan& p, const Bufs& f, cudaStream_t s);
cudaError_t launch_param_reduce(const Plan& p, const Bufs& f, cudaStream_t s);

int device_sm_count();

// Tensor-core variants (bf16, headdim 64); the launchers above use them when
// the problem is inside their supported set.
bool chunk_state_tc_supported(const Plan& p);
cudaError_t launch_chunk_state_tc(const Plan& p, const Bufs& f, bool dstates, cudaStream_t s);
bool chunk_scan_tc_supported(const Plan& p);
cudaError_t launch_chunk_scan_tc(const Plan& p, const Bufs& f, cudaStream_t s);
bool chunk_bwd_tc_supported(const Plan& p);
cudaError_t launch_chunk_bwd_tc(const Plan& p, const Bufs& f, cudaStream_t s);

// Single-pass forward (one persistent CTA per (batch row, head) chain, the
// carry kept on chip): bf16, headdim 64, d_state 64 or 128.
bool ssd_fwd_fused_supported(const Plan& p);
cudaError_t launch_ssd_fwd_fused(const Plan& p, const Bufs& f, cudaStream_t s);
// The backward's forward and reverse state chains, one CTA per chain
// (writes H_in, or dS with dinit and the dL/da_c partials).
bool state_chain_supported(const Plan& p);
cudaError_t launch_state_chain(const Plan& p, const Bufs& f, bool reverse, cudaStream_t s);

// Per-kernel timing hooks (ssd_profile.cu): each launcher names the kernel it
// launches; the entry points bracket every launch with prof_before/after.
void set_kernel_name(const char* name);
void prof_before(cudaStream_t s);
void prof_after(cudaStream_t s);

}  // namespace ssd
