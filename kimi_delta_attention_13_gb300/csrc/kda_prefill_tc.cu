// kda_prefill_tc.cu -- tensor-core chunked KDA prefill for sm_103a (bf16 in, fp32 state).
#include "kda_internal.cuh"

namespace kda {
namespace {
__device__ int g_prefill_tc_error;  // sticky device error word of this translation unit
}  // namespace

int read_and_clear_status_prefill_tc(cudaStream_t s, int32_t *status)
{
    int host = 0, zero = 0;
    if (cudaMemcpyFromSymbolAsync(&host, g_prefill_tc_error, sizeof(int), 0,
                                  cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return KDA_ERR_CUDA;
    if (cudaMemcpyToSymbolAsync(g_prefill_tc_error, &zero, sizeof(int), 0,
                                cudaMemcpyHostToDevice, s) != cudaSuccess)
        return KDA_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return KDA_ERR_CUDA;
    *status = host;
    return KDA_OK;
}

int launch_prefill_tc(const void *q, const void *k, const void *v, const void *g,
                      const void *beta, const int32_t *cu_seqlens, int n_seqs,
                      int64_t total_tokens, int n_heads, int out_dtype, const float *init_state,
                      void *out, float *final_state, int ckpt_stride, float *ckpts,
                      cudaStream_t stream)
{
    return launch_prefill_recurrent(q, k, v, g, beta, cu_seqlens, n_seqs, total_tokens, n_heads,
                                    128, 128, KDA_BF16, out_dtype, init_state, out, final_state,
                                    ckpt_stride, ckpts, stream);
}

}  // namespace kda
