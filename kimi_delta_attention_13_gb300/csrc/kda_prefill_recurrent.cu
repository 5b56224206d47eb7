// kda_prefill_recurrent.cu -- token-by-token KDA prefill on CUDA cores (fp32 state).
//
// Evaluates the recurrence of "Kimi K3 im Detail", section "Sequenz-Mixing: KDA-Zustand und
// globale MLA", in token order with the state in registers:
//     S' = diag(exp(clamp(g_t,-5,0))) S,  r = S'^T k_t,  S = S' + beta_t k_t (v_t - r)^T,
//     o_t = S^T q_t  (after the write).
// It is the fp32 path of kda_prefill and a second, independent evaluation of the bf16 path.
//
// Grid: one block per (sequence, head, 32-wide slice of the value channels); value columns
// are independent given k, g, beta, so slices never exchange data.  Block = 4 warps; in warp w,
// lane l owns column j = 8w + (l & 7) of the slice and the key rows i = 16 g + 4 (l >> 3) + c
// (g = 0..7, c = 0..3): four consecutive rows per group, read from shared memory as one float4,
// and the column sums over i are two xor-shuffles.  Tokens are staged 16 at a time in shared
// memory, by fully unrolled loops so that each thread's global loads of a stage are in flight
// together.
#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int kThreads = 128;
constexpr int kSlice = 32;         // value columns per block
constexpr int kMaxDk = 128;
constexpr int kRows = kMaxDk / 4;  // key rows per thread
constexpr int kStage = 16;         // tokens staged per shared-memory fill

template <typename T, typename TO>
__global__ void __launch_bounds__(kThreads)
prefill_recurrent_kernel(const T *__restrict__ q, const T *__restrict__ k, const T *__restrict__ v,
                         const T *__restrict__ g, const T *__restrict__ beta,
                         const int32_t *__restrict__ cu_seqlens, int64_t total_tokens, int H,
                         int dk, int dv, const float *__restrict__ init, TO *__restrict__ out,
                         float *__restrict__ final_state, int ckpt_stride, float *__restrict__ ckpts)
{
    const int n_slices = dv / kSlice;
    const int slice = blockIdx.x % n_slices;
    const int h = (blockIdx.x / n_slices) % H;
    const int n = blockIdx.x / (n_slices * H);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int jj = warp * 8 + (lane & 7);   // column inside the slice
    const int j = slice * kSlice + jj;      // value channel
    const int iq = lane >> 3;               // row phase: rows i = 4m + iq

    __shared__ __align__(16) float s_k[kStage][kMaxDk], s_q[kStage][kMaxDk], s_a[kStage][kMaxDk];
    __shared__ float s_v[kStage][kSlice];
    __shared__ float s_b[kStage];
    __shared__ int64_t s_first_ckpt;

    const int64_t start = cu_seqlens ? cu_seqlens[n] : 0;
    const int64_t end = cu_seqlens ? cu_seqlens[n + 1] : total_tokens;

    if (tid == 0) {  // first checkpoint slot of this sequence
        int64_t first = 0;
        if (ckpt_stride > 0 && cu_seqlens)
            for (int m = 0; m < n; ++m) first += (cu_seqlens[m + 1] - cu_seqlens[m]) / ckpt_stride;
        s_first_ckpt = first;
    }

    const int64_t sbase = ((int64_t)n * H + h) * dk * dv;
    float S[kRows];
#pragma unroll
    for (int m = 0; m < kRows; ++m) {
        const int i = 16 * (m >> 2) + 4 * iq + (m & 3);
        S[m] = (init && i < dk) ? init[sbase + (int64_t)i * dv + j] : 0.f;
    }

    const int64_t row_stride_k = (int64_t)H * dk, row_stride_v = (int64_t)H * dv;
    for (int64_t t0 = start; t0 < end; t0 += kStage) {
        const int cnt = (int)((end - t0) < kStage ? (end - t0) : kStage);
        __syncthreads();  // previous stage fully consumed
#pragma unroll 16
        for (int e = tid; e < kStage * kMaxDk; e += kThreads) {
            const int r = e / kMaxDk, c = e % kMaxDk;
            float kv = 0.f, qv = 0.f, av = 1.f;
            if (r < cnt && c < dk) {
                const int64_t off = (t0 + r) * row_stride_k + (int64_t)h * dk + c;
                kv = to_f32(k[off]);
                qv = to_f32(q[off]);
                av = retention(to_f32(g[off]));
            }
            s_k[r][c] = kv; s_q[r][c] = qv; s_a[r][c] = av;
        }
#pragma unroll
        for (int e = tid; e < kStage * kSlice; e += kThreads) {
            const int r = e / kSlice, c = e % kSlice;
            s_v[r][c] = r < cnt ? to_f32(v[(t0 + r) * row_stride_v + (int64_t)h * dv + slice * kSlice + c]) : 0.f;
        }
        if (tid < kStage) s_b[tid] = tid < cnt ? to_f32(beta[(t0 + tid) * H + h]) : 0.f;
        __syncthreads();

        for (int r = 0; r < cnt; ++r) {
            float rp = 0.f;
            float4 kr[kRows / 4];
#pragma unroll
            for (int gq = 0; gq < kRows / 4; ++gq) {
                const int i0 = 16 * gq + 4 * iq;
                const float4 a4 = *reinterpret_cast<const float4 *>(&s_a[r][i0]);
                kr[gq] = *reinterpret_cast<const float4 *>(&s_k[r][i0]);
                S[4 * gq + 0] *= a4.x; S[4 * gq + 1] *= a4.y; S[4 * gq + 2] *= a4.z; S[4 * gq + 3] *= a4.w;
                rp += S[4 * gq + 0] * kr[gq].x;
                rp += S[4 * gq + 1] * kr[gq].y;
                rp += S[4 * gq + 2] * kr[gq].z;
                rp += S[4 * gq + 3] * kr[gq].w;
            }
            rp += __shfl_xor_sync(0xffffffffu, rp, 8);
            rp += __shfl_xor_sync(0xffffffffu, rp, 16);
            const float u = s_b[r] * (s_v[r][jj] - rp);
            float op = 0.f;
#pragma unroll
            for (int gq = 0; gq < kRows / 4; ++gq) {
                const float4 q4 = *reinterpret_cast<const float4 *>(&s_q[r][16 * gq + 4 * iq]);
                S[4 * gq + 0] += kr[gq].x * u; S[4 * gq + 1] += kr[gq].y * u;
                S[4 * gq + 2] += kr[gq].z * u; S[4 * gq + 3] += kr[gq].w * u;
                op += S[4 * gq + 0] * q4.x;
                op += S[4 * gq + 1] * q4.y;
                op += S[4 * gq + 2] * q4.z;
                op += S[4 * gq + 3] * q4.w;
            }
            op += __shfl_xor_sync(0xffffffffu, op, 8);
            op += __shfl_xor_sync(0xffffffffu, op, 16);
            const int64_t t = t0 + r;
            if (iq == 0) store_as(out + t * row_stride_v + (int64_t)h * dv + j, op);
            const int64_t count = t - start + 1;
            if (ckpt_stride > 0 && count % ckpt_stride == 0) {
                const int64_t slot = s_first_ckpt + count / ckpt_stride - 1;
                float *dst = ckpts + (slot * H + h) * (int64_t)dk * dv;
#pragma unroll
                for (int m = 0; m < kRows; ++m) {
                    const int i = 16 * (m >> 2) + 4 * iq + (m & 3);
                    if (i < dk) dst[(int64_t)i * dv + j] = S[m];
                }
            }
        }
    }
    if (final_state) {
#pragma unroll
        for (int m = 0; m < kRows; ++m) {
            const int i = 16 * (m >> 2) + 4 * iq + (m & 3);
            if (i < dk) final_state[sbase + (int64_t)i * dv + j] = S[m];
        }
    }
}

}  // namespace

int launch_prefill_recurrent(const void *q, const void *k, const void *v, const void *g,
                             const void *beta, const int32_t *cu_seqlens, int n_seqs,
                             int64_t total_tokens, int n_heads, int d_k, int d_v, int dtype,
                             int out_dtype, const float *init_state, void *out, float *final_state,
                             int ckpt_stride, float *ckpts, cudaStream_t stream)
{
    if (d_k < 1 || d_k > kMaxDk || d_v < kSlice || d_v > 256 || d_v % kSlice != 0)
        return KDA_ERR_UNSUPPORTED_SHAPE;
    const int64_t blocks = (int64_t)n_seqs * n_heads * (d_v / kSlice);
    if (blocks == 0) return KDA_OK;
    if (blocks > 0x7fffffffLL) return KDA_ERR_INVALID_ARG;
    auto go = [&](auto in_tag, auto out_tag) {
        using T = decltype(in_tag);
        using TO = decltype(out_tag);
        prefill_recurrent_kernel<T, TO><<<(unsigned)blocks, kThreads, 0, stream>>>(
            (const T *)q, (const T *)k, (const T *)v, (const T *)g, (const T *)beta, cu_seqlens,
            total_tokens, n_heads, d_k, d_v, init_state, (TO *)out, final_state, ckpt_stride, ckpts);
    };
    if (dtype == KDA_BF16) {
        if (out_dtype == KDA_BF16) go(__nv_bfloat16{}, __nv_bfloat16{}); else go(__nv_bfloat16{}, float{});
    } else {
        if (out_dtype == KDA_BF16) go(float{}, __nv_bfloat16{}); else go(float{}, float{});
    }
    return cudaGetLastError() == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

}  // namespace kda
