// kda_internal.cuh -- helpers shared by the CUDA translation units of libkda_gb300.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/kda.h"

namespace kda {

// Element conversions for the two input/output dtypes.
__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ void store_as(float *p, float x) { *p = x; }
__device__ __forceinline__ void store_as(__nv_bfloat16 *p, float x) { *p = __float2bfloat16_rn(x); }

// Retention factor of one token for one key channel: exp of the log-decay clamped to the
// published range [-5, 0] ("Kimi K3 im Detail", section "Sequenz-Mixing", log-decay floor).
__device__ __forceinline__ float retention(float g) { return expf(fminf(fmaxf(g, -5.0f), 0.0f)); }

__host__ __device__ constexpr int ceil_div(int a, int b) { return (a + b - 1) / b; }

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Per-translation-unit readers of the sticky device error words (see kda_device_status).
int read_and_clear_status_state_copy(cudaStream_t s, int32_t *status);
int read_and_clear_status_prefill_tc(cudaStream_t s, int32_t *status);
int read_and_clear_status_prefill_tc_precise(cudaStream_t s, int32_t *status);
int read_and_clear_status_decode(cudaStream_t s, int32_t *status);
int read_and_clear_status_cp(cudaStream_t s, int32_t *status);
// Launch the one-CTA probe whose bounded device wait expires after `cycles` SM cycles.
int launch_wait_timeout_probe(long long cycles, cudaStream_t stream);
// Launch the one-thread run of the shared-memory bounds check on an out-of-window offset; read
// (and clear) the site number of the first failed bounds check.
int launch_bounds_check_probe(cudaStream_t stream);
int read_and_clear_debug_site(cudaStream_t s, int32_t *site);
int read_and_clear_debug_site_precise(cudaStream_t s, int32_t *site);

// Kernel launchers (host side, no validation: the C ABI validates first).
int launch_decode(const void *q, const void *k, const void *v, const void *g, const void *beta,
                  float *state, void *out, int n_seqs, int n_heads, int d_k, int d_v, int dtype,
                  int out_dtype, cudaStream_t stream);
int launch_state_copy(float *dst, const int64_t *dst_idx, int64_t n_dst, const float *src,
                      const int64_t *src_idx, int64_t n_src, int64_t n, int64_t unit_floats,
                      cudaStream_t stream);
int launch_prefill_recurrent(const void *q, const void *k, const void *v, const void *g,
                             const void *beta, const int32_t *cu_seqlens, int n_seqs,
                             int64_t total_tokens, int n_heads, int d_k, int d_v, int dtype,
                             int out_dtype, const float *init_state, void *out, float *final_state,
                             int ckpt_stride, float *ckpts, cudaStream_t stream);
int launch_premix(const void *xq, const void *xk, const void *xv, const void *a, const void *b,
                  const float *w, const void *hist, const int32_t *cu_seqlens, int n_seqs,
                  long long total_tokens, int n_heads, int d, float eps, int dtype, void *q,
                  void *k, void *v, void *g, void *beta, cudaStream_t stream);
int launch_output_gate(const void *o, int o_dtype, const void *z, int z_dtype, void *out,
                       int out_dtype, long long n, cudaStream_t stream);
int launch_cp_correct(const float *u, const float *s_start, const int32_t *cu_seg, int n_seg,
                      const int32_t *skip_seg, int n_skip, int H, long long T, float *out,
                      cudaStream_t stream);
int launch_cp_combine(const float *s_loc, const float *m, const int32_t *seq_seg, int n_seqs, int H,
                      float *s_start, float *final_state, cudaStream_t stream);
int64_t staged_scratch_ints(const int32_t *h_cu, int n_seqs, long long T, long long chunk_tokens);
int run_prefill_staged(const void *const h_in[5], const int32_t *h_cu, int n_seqs, long long T,
                       int H, int dtype, int out_dtype, const float *init_state, void *const d_in[5],
                       void *d_out, void *h_out, float *final_state, int32_t *d_scratch,
                       long long chunk_tokens, cudaStream_t stream);
int run_prefill_staged_static(const void *const h_in[5], const int32_t *h_cu, int n_seqs, long long T,
                              int H, int dtype, int out_dtype, const float *init_state,
                              void *const d_in[5], void *d_out, void *h_out, float *final_state,
                              long long chunk_tokens, cudaStream_t stream);
// streams and events the staged calls have created so far in this process
long long staged_handles_created();
int launch_prefill_tc(const void *q, const void *k, const void *v, const void *g,
                      const void *beta, const int32_t *cu_seqlens, int n_seqs,
                      int64_t total_tokens, int n_heads, int out_dtype, const float *init_state,
                      void *out, float *final_state, int ckpt_stride, float *ckpts,
                      cudaStream_t stream);
// the same kernel in its precise mode (Aqk carried in two fp16 parts)
int launch_prefill_tc_precise(const void *q, const void *k, const void *v, const void *g,
                              const void *beta, const int32_t *cu_seqlens, int n_seqs,
                              int64_t total_tokens, int n_heads, int out_dtype,
                              const float *init_state, void *out, float *final_state,
                              int ckpt_stride, float *ckpts, cudaStream_t stream);

}  // namespace kda
