// kda_cp.cu -- the scan that joins independently prefilled segments of a sequence
// (context-parallel prefill).
//
// Per token the recurrence ("Kimi K3 im Detail", section "Sequenz-Mixing: KDA-Zustand und globale
// MLA") is affine in the state: S_t = A_t S_(t-1) + beta_t k_t v_t^T with A_t =
// (I - beta_t k_t k_t^T) diag(exp(g_t)).  Over a segment, S_end = M S_start + S_loc, where S_loc is
// the segment prefilled from a zero state and M = A_L ... A_1 is the segment prefilled with v = 0
// from the identity.  Given those per segment, the scan
//     S_start(j + 1) = M(j) S_start(j) + S_loc(j)
// gives every segment's true start state, from which one more prefill of the segments produces
// the true outputs.
//
// The state's d_v columns are independent (M acts from the left), so the scan of one
// (sequence, head) is cut into 16 CTAs of 8 columns each.  A CTA keeps its 128 x 8 slice of the
// running state in registers (4 values per thread) and a copy in shared memory for the product's
// reads; the segment maps M(j), which do not depend on the chain, stream through a double buffer
// in shared memory with cp.async, M(j + 1) landing while M(j) is applied.  The 16 CTAs of a head
// are adjacent in the grid, so each M is read from HBM about once and from L2 by the rest.
// The arithmetic is fp32 FMA over k = 0 .. 127 in order, then the add of S_loc.
#include "kda_internal.cuh"
#include "sm100_ptx.cuh"

namespace kda {
namespace {

constexpr int kD = 128;                    // d_k = d_v
constexpr int kSlice = 8;                  // state columns per CTA
constexpr int kSlices = kD / kSlice;       // CTAs per (sequence, head)
constexpr int kScanThreads = 256;          // thread t: row t / 2, columns 4 (t % 2) .. + 3 of the slice
constexpr int kMStride = kD + 4;           // padded row of M in shared memory: rows r and r + 1
                                           // start 4 banks apart, so float4 row reads do not collide
constexpr int kScanSmem = (2 * kD * kMStride + kD * kSlice) * 4;   // 139,264 B
static_assert(kScanThreads == 2 * kD, "two threads per state row");

__device__ __forceinline__ void cp_async16(void *smem_dst, const void *gmem_src)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(ptx::smem_u32(smem_dst)), "l"(gmem_src)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// every committed group but the most recent one has landed (for this thread's own copies)
__device__ __forceinline__ void cp_async_wait_all_but_last()
{
    asm volatile("cp.async.wait_group 1;" ::: "memory");
}

// M (128 x 128 fp32, row-major, 16-byte aligned) into shared rows of kMStride floats
__device__ __forceinline__ void stage_m(float *dst, const float *src)
{
    for (int e = threadIdx.x; e < kD * kD / 4; e += kScanThreads)
        cp_async16(dst + (e >> 5) * kMStride + 4 * (e & 31), src + 4 * e);
}

// grid (kSlices * n_seqs, H): CTA (x, h) scans columns kSlice * (x % kSlices) .. + 7 of head h of
// sequence x / kSlices over its segments [seq_seg[n], seq_seg[n + 1])
__global__ void __launch_bounds__(kScanThreads) cp_combine_kernel(
    const float *__restrict__ s_loc, const float *__restrict__ m, const int32_t *__restrict__ seq_seg,
    int H, float *__restrict__ s_start, float *__restrict__ final_state)
{
    extern __shared__ __align__(16) float sm[];
    float *const sM0 = sm, *const sM1 = sm + kD * kMStride, *const sS = sm + 2 * kD * kMStride;
    const int n = blockIdx.x / kSlices, slice = blockIdx.x % kSlices, h = blockIdx.y;
    const int lo = seq_seg[n], hi = seq_seg[n + 1];
    if (hi <= lo) return;   // a sequence always has a segment; nothing to do otherwise
    const long long blk = (long long)kD * kD;
    const int row = threadIdx.x >> 1, half = 4 * (threadIdx.x & 1);
    const long long elem = row * kD + kSlice * slice + half;   // this thread's 4 values in a state
    // the running state: the end state of the first segment (prefilled from the sequence's own
    // initial state)
    float4 s = *reinterpret_cast<const float4 *>(s_loc + ((long long)lo * H + h) * blk + elem);
    if (lo + 1 < hi) stage_m(sM0, m + ((long long)(lo + 1) * H + h) * blk);
    cp_async_commit();
    for (int j = lo + 1; j < hi; ++j) {
        const long long off = ((long long)j * H + h) * blk;
        float *const cur = ((j - lo - 1) & 1) ? sM1 : sM0;
        float *const nxt = ((j - lo - 1) & 1) ? sM0 : sM1;
        // nxt was last read in the previous step, before its closing barrier
        if (j + 1 < hi) stage_m(nxt, m + ((long long)(j + 1) * H + h) * blk);
        cp_async_commit();
        *reinterpret_cast<float4 *>(s_start + off + elem) = s;
        *reinterpret_cast<float4 *>(sS + row * kSlice + half) = s;
        const float4 l = *reinterpret_cast<const float4 *>(s_loc + off + elem);
        cp_async_wait_all_but_last();
        __syncthreads();   // M(j) and the slice of S_start(j) are in shared memory
        const float *mr = cur + row * kMStride;
        const float *sc = sS + half;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
        for (int k = 0; k < kD; k += 4) {
            const float4 a = *reinterpret_cast<const float4 *>(mr + k);
            const float av[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                const float4 b = *reinterpret_cast<const float4 *>(sc + (k + kk) * kSlice);
                acc.x = fmaf(av[kk], b.x, acc.x);
                acc.y = fmaf(av[kk], b.y, acc.y);
                acc.z = fmaf(av[kk], b.z, acc.z);
                acc.w = fmaf(av[kk], b.w, acc.w);
            }
        }
        __syncthreads();   // every thread is done with sS and with cur
        s = make_float4(acc.x + l.x, acc.y + l.y, acc.z + l.z, acc.w + l.w);
    }
    if (final_state)
        *reinterpret_cast<float4 *>(final_state + ((long long)n * H + h) * blk + elem) = s;
}

}  // namespace

int launch_cp_combine(const float *s_loc, const float *m, const int32_t *seq_seg, int n_seqs, int H,
                      float *s_start, float *final_state, cudaStream_t stream)
{
    if (n_seqs == 0) return KDA_OK;
    if ((long long)n_seqs * kSlices > 0x7fffffffLL || H > 65535) return KDA_ERR_UNSUPPORTED_SHAPE;
    if (cudaFuncSetAttribute(cp_combine_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kScanSmem) != cudaSuccess)
        return KDA_ERR_CUDA;
    cp_combine_kernel<<<dim3(kSlices * n_seqs, H), kScanThreads, kScanSmem, stream>>>(
        s_loc, m, seq_seg, H, s_start, final_state);
    return cudaGetLastError() == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

}  // namespace kda
