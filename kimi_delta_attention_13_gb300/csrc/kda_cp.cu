// kda_cp.cu -- the scan that joins independently prefilled segments of a sequence
// (context-parallel prefill).
//
// Per token the recurrence ("Kimi K3 im Detail", section "Sequenz-Mixing: KDA-Zustand und globale
// MLA") is affine in the state: S_t = A_t S_(t-1) + beta_t k_t v_t^T with A_t =
// (I - beta_t k_t k_t^T) diag(exp(g_t)).  Over a segment, S_end = M S_start + S_loc, where S_loc is
// the segment prefilled from a zero state and M = A_L ... A_1 is the segment prefilled with v = 0
// from the identity.  Given those per segment, the scan
//     S_start(j) = M(j-1) S_start(j-1) + S_loc(j-1)
// gives every segment's true start state, from which one more prefill of the segments produces
// the true outputs.  The scan runs one CTA per (sequence, head): fp32 128 x 128 products on CUDA
// cores, with M and the running state staged in shared memory.
#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int kD = 128;            // d_k = d_v
constexpr int kCpThreads = 512;
constexpr int kCombineSmem = 2 * kD * kD * 4;   // M and S: 128 KB

// the scan for one (sequence, head) over its segments [seq_seg[n], seq_seg[n+1])
__global__ void __launch_bounds__(kCpThreads) cp_combine_kernel(
    const float *__restrict__ s_loc, const float *__restrict__ m, const int32_t *__restrict__ seq_seg,
    int H, float *__restrict__ s_start, float *__restrict__ final_state)
{
    extern __shared__ __align__(16) float sm[];
    float *sM = sm, *sS = sm + kD * kD;
    const int n = blockIdx.x, h = blockIdx.y;
    const int lo = seq_seg[n], hi = seq_seg[n + 1];
    const long long blk = (long long)kD * kD;
    if (hi <= lo) return;   // a sequence always has a segment; nothing to do otherwise
    // thread (rg, cg): rows 8 rg .. 8 rg + 7, columns 4 cg .. 4 cg + 3 of the 128 x 128 product
    const int cg = threadIdx.x & 31, rg = threadIdx.x >> 5;
    // S = end state of the first segment (prefilled from the sequence's own initial state)
    const float4 *first = reinterpret_cast<const float4 *>(s_loc + ((long long)lo * H + h) * blk);
    for (int e = threadIdx.x; e < kD * kD / 4; e += kCpThreads) reinterpret_cast<float4 *>(sS)[e] = first[e];
    for (int j = lo + 1; j < hi; ++j) {
        const long long off = ((long long)j * H + h) * blk;
        const float4 *mj = reinterpret_cast<const float4 *>(m + off);
        float4 *dst = reinterpret_cast<float4 *>(s_start + off);
        __syncthreads();   // sS holds S_start(j)
        for (int e = threadIdx.x; e < kD * kD / 4; e += kCpThreads) {
            dst[e] = reinterpret_cast<const float4 *>(sS)[e];
            reinterpret_cast<float4 *>(sM)[e] = mj[e];
        }
        __syncthreads();
        float acc[8][4];
#pragma unroll
        for (int r = 0; r < 8; ++r)
#pragma unroll
            for (int c = 0; c < 4; ++c) acc[r][c] = 0.f;
        for (int kk = 0; kk < kD; ++kk) {
            const float4 b = *reinterpret_cast<const float4 *>(sS + kk * kD + 4 * cg);
#pragma unroll
            for (int r = 0; r < 8; ++r) {
                const float a = sM[(8 * rg + r) * kD + kk];
                acc[r][0] = fmaf(a, b.x, acc[r][0]);
                acc[r][1] = fmaf(a, b.y, acc[r][1]);
                acc[r][2] = fmaf(a, b.z, acc[r][2]);
                acc[r][3] = fmaf(a, b.w, acc[r][3]);
            }
        }
        __syncthreads();   // every thread has read sS
        const float *lj = s_loc + off;
#pragma unroll
        for (int r = 0; r < 8; ++r) {
            const int row = 8 * rg + r;
            const float4 l = *reinterpret_cast<const float4 *>(lj + row * kD + 4 * cg);
            *reinterpret_cast<float4 *>(sS + row * kD + 4 * cg) =
                make_float4(acc[r][0] + l.x, acc[r][1] + l.y, acc[r][2] + l.z, acc[r][3] + l.w);
        }
    }
    __syncthreads();
    if (final_state) {
        float4 *dst = reinterpret_cast<float4 *>(final_state + ((long long)n * H + h) * blk);
        for (int e = threadIdx.x; e < kD * kD / 4; e += kCpThreads) dst[e] = reinterpret_cast<const float4 *>(sS)[e];
    }
}

}  // namespace

int launch_cp_combine(const float *s_loc, const float *m, const int32_t *seq_seg, int n_seqs, int H,
                      float *s_start, float *final_state, cudaStream_t stream)
{
    if (n_seqs == 0) return KDA_OK;
    if (cudaFuncSetAttribute(cp_combine_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kCombineSmem) != cudaSuccess)
        return KDA_ERR_CUDA;
    cp_combine_kernel<<<dim3(n_seqs, H), kCpThreads, kCombineSmem, stream>>>(s_loc, m, seq_seg, H,
                                                                             s_start, final_state);
    return cudaGetLastError() == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

}  // namespace kda
