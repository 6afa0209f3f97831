// k_shard.cu -- the joins of context parallelism: a sequence split into
// contiguous shards (one per rank), each shard run on its own through
// ssd_fwd / ssd_bwd, the shards joined by exclusive folds of per-shard pairs.
//
// Page "B200 Helion Mamba-2" (aitrends.kr/articles/109906), integration
// plans: context parallelism (the sequence sharded across ranks) is the
// extension the drop-in module is meant to support; the page gives no
// method.  It follows from the recurrence (page "llm-mamba-200", sections
// 2-3): a shard maps the state h entering it to dec * h + final(0), with dec
// the product of its per-token decays exp(dt_eff * A) -- 0 when a new
// sequence starts after the shard's first token -- and final(0) its final
// state from a zero start.  These pairs compose with the chunk operator
// (a, b) o (a', b') = (a a', a' b + b'), so one left-to-right fold gives
// every shard its entering state (zero when its first token starts a new
// sequence).  The backward mirrors it right to left: a shard's
// dinitial_states is affine in the gradient g at its final state,
// dinit(g) = dec * g + dinit(0).
//
//   shard_decay_kernel: one warp per (row, head): the shard's sum of
//     dt_eff * A (fixed-order: lane-strided partial sums, then a shuffle
//     tree), exp of it, or 0 on a sequence start inside the shard; also the
//     segment ids of the shard's first and last tokens per row.
//   shard_fold_kernel: one thread per (row, head, state element), the fold
//     over the shards in order (or in reverse), coalesced over the state
//     elements.
#include "ssd_internal.cuh"

namespace ssd {

namespace {

__device__ __forceinline__ float softplus_f(float z) { return fmaxf(z, 0.0f) + log1pf(expf(-fabsf(z))); }

template <typename T>
__global__ void __launch_bounds__(256) shard_decay_kernel(int b, int L, int H, const T* dt, const float* dt_bias,
                                                          const float* A, const int32_t* seq, float* decay,
                                                          int32_t* first_id, int32_t* last_id) {
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  if (warp >= b * H) return;
  const int bi = warp / H, h = warp % H;
  const float bias = dt_bias[h], Ah = A[h];
  float sum = 0.0f;
  int brk = 0;
  for (int t = lane; t < L; t += 32) {
    sum += softplus_f(to_f(dt[((long long)bi * L + t) * H + h]) + bias);
    if (seq != nullptr && t > 0 && seq[(long long)bi * L + t] != seq[(long long)bi * L + t - 1]) brk = 1;
  }
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) {
    sum += __shfl_xor_sync(0xffffffffu, sum, d);
    brk |= __shfl_xor_sync(0xffffffffu, brk, d);
  }
  if (lane == 0) {
    decay[warp] = brk ? 0.0f : expf(sum * Ah);
    if (h == 0 && first_id != nullptr) {
      first_id[bi] = seq != nullptr ? seq[(long long)bi * L] : 0;
      last_id[bi] = seq != nullptr ? seq[(long long)bi * L + L - 1] : 0;
    }
  }
}

// Forward:  h = boundary (or 0); for r: [r > 0 and shard r starts a new
//           sequence] h = 0;  out[r] = h;  h = dec[r] h + local[r];  total = h.
// Reverse:  g = boundary (or 0); for r = R-1 .. 0: out[r] = g;
//           g = dec[r] g + local[r];  [r > 0 and shard r starts a new
//           sequence] g = 0;  total = g.
template <bool kRev>
__global__ void __launch_bounds__(256) shard_fold_kernel(int R, int b, int H, int PN, const float* decay,
                                                         const float* local, const int32_t* first_id,
                                                         const int32_t* last_id, const float* boundary,
                                                         float* out, float* total) {
  const long long per = (long long)b * H * PN;
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= per) return;
  const long long bh = i / PN;
  const int bi = (int)(bh / H);
  auto starts_new = [&](int r) {
    return r > 0 && first_id != nullptr && first_id[(long long)r * b + bi] != last_id[(long long)(r - 1) * b + bi];
  };
  float v = boundary != nullptr ? boundary[i] : 0.0f;
  for (int k = 0; k < R; ++k) {
    const int r = kRev ? R - 1 - k : k;
    if (!kRev && starts_new(r)) v = 0.0f;
    out[(long long)r * per + i] = v;
    v = fmaf(decay[(long long)r * b * H + bh], v, local[(long long)r * per + i]);
    if (kRev && starts_new(r)) v = 0.0f;
  }
  if (total != nullptr) total[i] = v;
}

bool aligned16(const void* p) { return p == nullptr || (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

int device_check();

}  // namespace ssd

using namespace ssd;

extern "C" int ssd_shard_decay(const ssd_problem* prob, const void* dt, const float* dt_bias, const float* A,
                               const int32_t* seq_idx, float* decay, int32_t* first_ids, int32_t* last_ids,
                               ssd_stream_t stream) {
  if (!prob || !dt || !dt_bias || !A || !decay) return SSD_ERR_INVALID_ARGUMENT;
  if (prob->batch < 1 || prob->seqlen < 1 || prob->nheads < 1 || prob->batch > 65535 || prob->nheads > 65535)
    return SSD_ERR_INVALID_ARGUMENT;
  if (prob->dtype != SSD_F32 && prob->dtype != SSD_BF16) return SSD_ERR_INVALID_ARGUMENT;
  if (((prob->flags & SSD_HAS_SEQ_IDX) != 0) != (seq_idx != nullptr)) return SSD_ERR_INVALID_ARGUMENT;
  if ((first_ids == nullptr) != (last_ids == nullptr)) return SSD_ERR_INVALID_ARGUMENT;
  if (prob->seqlen > (int64_t(1) << 30) || prob->batch * prob->nheads > (int64_t(1) << 26))
    return SSD_ERR_UNSUPPORTED;
  const int rc = device_check();
  if (rc != SSD_OK) return rc;
  const int b = (int)prob->batch, L = (int)prob->seqlen, H = (int)prob->nheads;
  const long long warps = (long long)b * H;
  const int blocks = (int)((warps * 32 + 255) / 256);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  set_kernel_name("shard_decay");
  prof_before(s);
  if (prob->dtype == SSD_BF16)
    shard_decay_kernel<__nv_bfloat16><<<blocks, 256, 0, s>>>(b, L, H, static_cast<const __nv_bfloat16*>(dt),
                                                             dt_bias, A, seq_idx, decay, first_ids, last_ids);
  else
    shard_decay_kernel<float><<<blocks, 256, 0, s>>>(b, L, H, static_cast<const float*>(dt), dt_bias, A,
                                                     seq_idx, decay, first_ids, last_ids);
  const cudaError_t e = cudaGetLastError();
  prof_after(s);
  return e == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}

extern "C" int ssd_shard_fold(int64_t nshards, int64_t batch, int64_t nheads, int64_t headdim, int64_t dstate,
                              const float* decay, const float* local, const int32_t* first_ids,
                              const int32_t* last_ids, const float* boundary, float* out, float* total,
                              int reverse, ssd_stream_t stream) {
  if (nshards < 1 || batch < 1 || nheads < 1 || headdim < 1 || dstate < 1) return SSD_ERR_INVALID_ARGUMENT;
  if (!decay || !local || !out) return SSD_ERR_INVALID_ARGUMENT;
  if ((first_ids == nullptr) != (last_ids == nullptr)) return SSD_ERR_INVALID_ARGUMENT;
  if (nshards > 65535 || batch > 65535 || nheads > 65535 || headdim * dstate > (int64_t(1) << 20))
    return SSD_ERR_UNSUPPORTED;
  const void* ptrs[] = {decay, local, first_ids, last_ids, boundary, out, total};
  for (const void* q : ptrs)
    if (!aligned16(q)) return SSD_ERR_INVALID_ARGUMENT;
  const int rc = device_check();
  if (rc != SSD_OK) return rc;
  const long long per = batch * nheads * headdim * dstate;
  if (per >= (int64_t(1) << 38)) return SSD_ERR_UNSUPPORTED;  // grid of at most 2^30 blocks
  const int blocks = (int)((per + 255) / 256);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  set_kernel_name(reverse ? "shard_fold_bwd" : "shard_fold_fwd");
  prof_before(s);
  const int R = (int)nshards, b = (int)batch, H = (int)nheads, PN = (int)(headdim * dstate);
  if (reverse)
    shard_fold_kernel<true><<<blocks, 256, 0, s>>>(R, b, H, PN, decay, local, first_ids, last_ids, boundary, out,
                                                   total);
  else
    shard_fold_kernel<false><<<blocks, 256, 0, s>>>(R, b, H, PN, decay, local, first_ids, last_ids, boundary,
                                                    out, total);
  const cudaError_t e = cudaGetLastError();
  prof_after(s);
  return e == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}
