// kda_cp.cu -- the scan that joins independently prefilled segments of a sequence
// (context-parallel prefill).
//
// Per token the recurrence ("Kimi K3 im Detail", section "Sequenz-Mixing: KDA-Zustand und globale
// MLA") is affine in the state: S_t = A_t S_(t-1) + beta_t k_t v_t^T with A_t =
// (I - beta_t k_t k_t^T) diag(exp(g_t)).  Over a segment, S_end = M S_start + S_loc, where S_loc is
// the segment prefilled from a zero state and M = A_L ... A_1 is the segment prefilled with v = 0
// from the identity.  Given those per segment, the scan
//     S_start(j + 1) = M(j) S_start(j) + S_loc(j)
// gives every segment's true start state.  The outputs follow without another prefill: with
// P_t = A_t ... A_1 (the segment's prefix map), the true state is S_t = P_t S_start + S_loc,t, so
//     o_t = S_t^T q_t = o_loc,t + S_start^T u_t,   u_t = P_t^T q_t,
// where o_loc,t are the outputs of the prefill from zeros and u_t those of the prefill with v = 0
// from the identity (S_t = P_t there).  kda_cp_correct adds S_start^T u_t to the outputs of every
// segment that does not start its sequence, as one tensor-core product per (segment, head).
//
// The state's d_v columns are independent (M acts from the left), so the scan of one
// (sequence, head) is cut into 16 CTAs of 8 columns each.  A CTA keeps its 128 x 8 slice of the
// running state in registers (4 values per thread) and a copy in shared memory for the product's
// reads; the segment maps M(j), which do not depend on the chain, stream through a double buffer
// in shared memory with cp.async, M(j + 1) landing while M(j) is applied.  The 16 CTAs of a head
// are adjacent in the grid, so each M is read from HBM about once and from L2 by the rest.
// The arithmetic is fp32 FMA over k = 0 .. 127 in order, then the add of S_loc.
#include <cudaTypedefs.h>

#include <mutex>

#include "kda_internal.cuh"
#include "sm100_ptx.cuh"

namespace kda {

__device__ int g_cp_error;   // sticky device error word of this translation unit

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


// ------------------------------------------------------------------------------------------------
// The output correction out_t += S_start^T u_t of one (segment, head), as D = A B on the tensor
// cores (kind::tf32, fp32 accumulation in TMEM):
//   A = S_start^T  M = 128 value channels j, K = 128 key channels m; staged once per CTA into
//                  shared memory, K-major (row j), rounded to nearest tf32;
//   B = u tile     K = 128, N = 128 tokens; K-major with one token per row, which is the layout
//                  of u itself, so TMA copies it in unchanged (128-byte swizzle);
//   D[j][t]        TMEM lane j, column t.  Thread j of an epilogue warp holds channel j of 32
//                  tokens, so each token's 128 outputs are read and written by 128 consecutive
//                  threads (512 contiguous bytes).
// Warp 0 lane 0 issues the TMA loads of u (a ring of two tiles) and the MMAs (two accumulators);
// warp 1 allocates TMEM; warps 4..11 add the accumulators to the outputs (warp w: the lanes of
// quarter w % 4, tokens 64 ((w - 4) / 4) .. + 63 of the tile).  Tokens of the tile past the
// segment's end are loaded (or zero past the tensor's end) and multiplied, but not written.
constexpr int kCorrTok = 128;                              // tokens per tile (MMA N)
constexpr int kCorrThreads = 384;
constexpr uint32_t kCorrRegion = 128 * 128;                // 128 rows x 32 fp32: one K slice
constexpr uint32_t kCorrTile = 4 * kCorrRegion;            // 128 x 128 fp32
constexpr uint32_t kCorrOffU = kCorrTile;                  // A first, then two u tiles
constexpr uint32_t kCorrOffShared = kCorrOffU + 2 * kCorrTile;
constexpr uint32_t kCorrSmem = kCorrOffShared + 128 + 1024;   // + barriers and flags; alignment
constexpr uint32_t kCorrCols = 2 * kCorrTok;               // TMEM columns: two accumulators
constexpr uint32_t kCorrIdesc = ptx::idesc_f32acc(128, kCorrTok, ptx::FMT_TF32, 0, 0);
constexpr long long kCorrTimeout = 2000000000ll;           // bounded waits: 2e9 SM cycles (~1 s)
static_assert(kCorrSmem <= 232448, "shared memory per block");

struct CorrShared {
    uint64_t full[2];        // u tile landed (TMA transaction bytes)
    uint64_t empty[2];       // the MMAs that read a u tile completed
    uint64_t acc_full[2];    // an accumulator holds its tile's product
    uint64_t acc_empty[2];   // the 8 epilogue warps read an accumulator
    uint64_t drain;          // end of the CTA: every MMA completed
    uint32_t tmem;
    int abort;
    int zero;                // always 0: the abort flag of waits that must not give up early
};
static_assert(sizeof(CorrShared) <= 128, "correction's shared block");

__device__ __forceinline__ uint64_t corr_desc_at(uint64_t d, uint32_t bytes) { return d + (bytes >> 4); }

__device__ __forceinline__ void corr_fail(CorrShared *sh)
{
    atomicExch(&g_cp_error, KDA_ERR_DEVICE_TIMEOUT);
    *reinterpret_cast<volatile int *>(&sh->abort) = 1;
}

// grid (n_seg, H): CTA (seg, h) corrects tokens [cu_seg[seg], cu_seg[seg + 1]) of head h, unless
// seg is one of the n_skip (increasing) indices skip_seg
__global__ void __launch_bounds__(kCorrThreads, 1) cp_correct_kernel(
    const __grid_constant__ CUtensorMap mu, const float *__restrict__ s_start,
    const int32_t *__restrict__ cu_seg, const int32_t *__restrict__ skip_seg, int n_skip, int H,
    float *__restrict__ out)
{
    using namespace ptx;
    extern __shared__ __align__(16) uint8_t corr_raw[];
    uint8_t *smem = corr_raw + ((1024u - (smem_u32(corr_raw) & 1023u)) & 1023u);
    CorrShared *sh = reinterpret_cast<CorrShared *>(smem + kCorrOffShared);
    const int seg = blockIdx.x, h = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // a segment that starts its sequence was prefilled from the sequence's own initial state, so
    // its outputs are already the true ones: such segments are listed in skip_seg
    {
        int lo = 0, hi = n_skip;
        while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            if (skip_seg[mid] < seg) lo = mid + 1; else hi = mid;
        }
        if (lo < n_skip && skip_seg[lo] == seg) return;
    }
    const long long t0 = cu_seg[seg], t1 = cu_seg[seg + 1];
    if (t1 <= t0) return;
    const int ntiles = (int)((t1 - t0 + kCorrTok - 1) / kCorrTok);

    if (threadIdx.x == 0) {
        for (int i = 0; i < 2; ++i) {
            mbar_init(&sh->full[i], 1);
            mbar_init(&sh->empty[i], 1);
            mbar_init(&sh->acc_full[i], 1);
            mbar_init(&sh->acc_empty[i], 8);
        }
        mbar_init(&sh->drain, 1);
        sh->abort = 0;
        sh->zero = 0;
        fence_barrier_init();
        tma_prefetch_desc(&mu);
    }
    if (warp == 1) {
        tmem_alloc(&sh->tmem, kCorrCols);
        tmem_relinquish();
    }
    // A = S_start^T: element (j, m) at K slice m / 32, row j; fp32 rounded to nearest tf32 by
    // adding half a tf32 ulp to the bit pattern (the product reads the top 19 bits)
    const float *S = s_start + ((long long)seg * H + h) * kD * kD;
    for (int e = threadIdx.x; e < kD * kD; e += kCorrThreads) {
        const int m = e >> 7, j = e & 127;
        *reinterpret_cast<uint32_t *>(smem + (m >> 5) * kCorrRegion + sw128(j, (m & 31) * 4)) =
            __float_as_uint(S[e]) + 0x1000u;
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tm = sh->tmem;

    if (warp == 0) {
        if (lane == 0) {
            const uint32_t sb = smem_u32(smem);
            const uint64_t a = smem_desc(sb, 0, 1024);
            int ld = 0, mm = 0;   // next tile to load, next tile to multiply
            long long last = clock64();
            while (mm < ntiles) {
                bool prog = false;
                // u tile `ld` into ring slot ld % 2, once the MMAs of tile ld - 2 have read it
                if (ld < ntiles && (ld < 2 || mbar_test_wait(&sh->empty[ld & 1], ((ld >> 1) - 1) & 1))) {
                    uint64_t *bar = &sh->full[ld & 1];
                    mbar_arrive_expect_tx(bar, kCorrTile);
                    for (int r = 0; r < 4; ++r)
                        tma_load_3d(smem + kCorrOffU + (ld & 1) * kCorrTile + r * kCorrRegion, &mu, bar,
                                    32 * r, h, (int)(t0 + (long long)ld * kCorrTok));
                    ++ld;
                    prog = true;
                }
                // tile `mm`: its u landed, and the epilogue read accumulator mm % 2 (tile mm - 2)
                if (mm < ld && mbar_test_wait(&sh->full[mm & 1], (mm >> 1) & 1) &&
                    (mm < 2 || mbar_test_wait(&sh->acc_empty[mm & 1], ((mm >> 1) - 1) & 1))) {
                    tc_fence_after();
                    const uint64_t b = smem_desc(sb + kCorrOffU + (mm & 1) * kCorrTile, 0, 1024);
#pragma unroll
                    for (int k = 0; k < 16; ++k)
                        mma_ss_tf32(tm + (mm & 1) * kCorrTok,
                                    corr_desc_at(a, (k >> 2) * kCorrRegion + (k & 3) * 32),
                                    corr_desc_at(b, (k >> 2) * kCorrRegion + (k & 3) * 32), kCorrIdesc, k > 0);
                    mma_commit(&sh->empty[mm & 1]);
                    mma_commit(&sh->acc_full[mm & 1]);
                    ++mm;
                    prog = true;
                }
                if (prog) {
                    last = clock64();
                } else {
                    if (*reinterpret_cast<volatile int *>(&sh->abort)) break;
                    if (clock64() - last > kCorrTimeout) {
                        corr_fail(sh);
                        break;
                    }
                    __nanosleep(32);
                }
            }
            // no copy or product in flight when the CTA leaves
            for (int t = mm; t < ld; ++t) mbar_wait(&sh->full[t & 1], (t >> 1) & 1, &sh->zero, kCorrTimeout);
            mma_commit(&sh->drain);
            mbar_wait(&sh->drain, 0, &sh->zero, kCorrTimeout);
        }
    } else if (warp >= 4) {
        const int q = warp & 3, hf = (warp - 4) >> 2;
        const uint32_t tq = tm + ((uint32_t)(32 * q) << 16);
        const long long rowstride = (long long)H * kD;
        for (int i = 0; i < ntiles; ++i) {
            if (!mbar_wait(&sh->acc_full[i & 1], (i >> 1) & 1, &sh->abort, kCorrTimeout)) {
                corr_fail(sh);
                break;
            }
            tc_fence_after();
#pragma unroll 1
            for (int c = 0; c < 64; c += 32) {
                const long long tb = t0 + (long long)i * kCorrTok + 64 * hf + c;
                uint32_t r[32];
                tmem_ld32(tq + (i & 1) * kCorrTok + 64 * hf + c, r);
                tmem_wait_ld();
                const long long left = t1 - tb;
                const int nvalid = left < 32 ? (int)left : 32;   // may be <= 0
                float *o = out + (tb * H + h) * kD + 32 * q + lane;
                float v[32];
#pragma unroll
                for (int x = 0; x < 32; ++x) v[x] = x < nvalid ? o[x * rowstride] : 0.f;
#pragma unroll
                for (int x = 0; x < 32; ++x)
                    if (x < nvalid) o[x * rowstride] = v[x] + __uint_as_float(r[x]);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sh->acc_empty[i & 1]);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tm, kCorrCols);
}

PFN_cuTensorMapEncodeTiled_v12000 corr_encode_fn()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    });
    return fn;
}

// u [T, H, 128] fp32: box = 32 channels (128 bytes) x 1 head x 128 tokens, 128-byte swizzle
bool make_u_map(CUtensorMap *map, const float *u, int H, long long T)
{
    auto enc = corr_encode_fn();
    if (!enc) return false;
    cuuint64_t dims[3] = {(cuuint64_t)kD, (cuuint64_t)H, (cuuint64_t)T};
    cuuint64_t strides[2] = {(cuuint64_t)kD * 4, (cuuint64_t)H * kD * 4};
    cuuint32_t box[3] = {32, 1, (cuuint32_t)kCorrTok}, es[3] = {1, 1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float *>(u), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
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

int launch_cp_correct(const float *u, const float *s_start, const int32_t *cu_seg, int n_seg,
                      const int32_t *skip_seg, int n_skip, int H, long long T, float *out, cudaStream_t stream)
{
    if (n_seg == 0 || T == 0) return KDA_OK;
    if (H > 65535 || T > 0x7fffffffLL) return KDA_ERR_UNSUPPORTED_SHAPE;
    CUtensorMap mu;
    if (!make_u_map(&mu, u, H, T)) return KDA_ERR_CUDA;
    if (cudaFuncSetAttribute(cp_correct_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kCorrSmem) != cudaSuccess)
        return KDA_ERR_CUDA;
    cp_correct_kernel<<<dim3(n_seg, H), kCorrThreads, kCorrSmem, stream>>>(mu, s_start, cu_seg, skip_seg,
                                                                            n_skip, H, out);
    return cudaGetLastError() == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

int read_and_clear_status_cp(cudaStream_t s, int32_t *status)
{
    int host = 0, zero = 0;
    if (cudaMemcpyFromSymbolAsync(&host, g_cp_error, sizeof(int), 0, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaMemcpyToSymbolAsync(g_cp_error, &zero, sizeof(int), 0, cudaMemcpyHostToDevice, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return KDA_ERR_CUDA;
    *status = host;
    return KDA_OK;
}

}  // namespace kda
