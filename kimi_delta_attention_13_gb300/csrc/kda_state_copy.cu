// kda_state_copy.cu -- indexed copy of whole per-sequence KDA states (checkpoint restore).
//
// Prefix reuse ("Kimi K3 im Detail", section "Sequenz-Mixing", prefix-reuse paragraph)
// restarts a sequence from a stored KDA state at the same token boundary as the global
// attention cache; this kernel moves such states between slot arrays:
//     dst[dst_idx[i]] = src[src_idx[i]],  one slot = H * d_k * d_v fp32.
// Pure HBM copy.  When a slot is a whole number of 16-byte units (always for d_k = d_v = 128), each
// block moves one 64 KB chunk of a slot by a 1-D bulk copy into shared memory and a bulk store out
// (three blocks per SM, so up to three chunks per SM in flight).  Otherwise 128-bit or scalar
// streaming loads and stores, four loads in flight per thread ahead of their stores.  Indices
// outside their slot range skip the copy and set this unit's sticky error word.
#include "kda_internal.cuh"
#include "sm100_ptx.cuh"

namespace kda {
namespace {

__device__ int g_state_copy_error;  // sticky device error word of this translation unit

template <typename V>
__global__ void __launch_bounds__(256)
state_copy_kernel(V *__restrict__ dst, const int64_t *__restrict__ dst_idx, int64_t n_dst,
                  const V *__restrict__ src, const int64_t *__restrict__ src_idx, int64_t n_src,
                  int64_t n, int64_t unit_vecs)
{
    constexpr int U = 4;   // loads in flight per thread before their stores
    for (int64_t i = blockIdx.y; i < n; i += gridDim.y) {
        const int64_t d = dst_idx ? dst_idx[i] : i;
        const int64_t s = src_idx ? src_idx[i] : i;
        if (d < 0 || d >= n_dst || s < 0 || s >= n_src) {
            if (threadIdx.x == 0 && blockIdx.x == 0) atomicExch(&g_state_copy_error, KDA_ERR_INDEX_RANGE);
            continue;
        }
        V *out = dst + d * unit_vecs;
        const V *in = src + s * unit_vecs;
        const int64_t stride = (int64_t)gridDim.x * blockDim.x;
        for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < unit_vecs; e += U * stride) {
            V v[U];
#pragma unroll
            for (int u = 0; u < U; ++u)
                if (e + u * stride < unit_vecs) v[u] = __ldcs(in + e + u * stride);
#pragma unroll
            for (int u = 0; u < U; ++u)
                if (e + u * stride < unit_vecs) __stcs(out + e + u * stride, v[u]);
        }
    }
}

constexpr uint32_t kChunkBytes = 65536;
constexpr long long kCopyTimeout = 2000000000ll;   // SM cycles (~1 s): bounded waits

// block b copies chunk b % chunks of slot pair b / chunks; lane 0 of the one warp does the work
__global__ void __launch_bounds__(32)
state_copy_bulk_kernel(char *__restrict__ dst, const int64_t *__restrict__ dst_idx, int64_t n_dst,
                       const char *__restrict__ src, const int64_t *__restrict__ src_idx,
                       int64_t n_src, int64_t unit_bytes, int64_t chunks)
{
    using namespace ptx;
    extern __shared__ __align__(128) uint8_t buf[];
    __shared__ __align__(8) uint64_t bar;
    __shared__ int s_zero;   // the abort flag of the waits: never set, they end by timeout only
    if (threadIdx.x != 0) return;
    const int64_t i = (int64_t)blockIdx.x / chunks, c = (int64_t)blockIdx.x % chunks;
    const int64_t d = dst_idx ? dst_idx[i] : i;
    const int64_t s = src_idx ? src_idx[i] : i;
    if (d < 0 || d >= n_dst || s < 0 || s >= n_src) {
        if (c == 0) atomicExch(&g_state_copy_error, KDA_ERR_INDEX_RANGE);
        return;
    }
    const int64_t off = c * kChunkBytes;
    const uint32_t bytes = (uint32_t)(unit_bytes - off < kChunkBytes ? unit_bytes - off : kChunkBytes);
    s_zero = 0;
    mbar_init(&bar, 1);
    fence_barrier_init();
    mbar_arrive_expect_tx(&bar, bytes);
    bulk_load_1d(buf, src + s * unit_bytes + off, bytes, &bar);
    if (!mbar_wait(&bar, 0, &s_zero, kCopyTimeout)) {
        atomicExch(&g_state_copy_error, KDA_ERR_DEVICE_TIMEOUT);
        mbar_wait(&bar, 0, &s_zero, kCopyTimeout);   // no copy left in flight at exit
        return;
    }
    bulk_store_1d(dst + d * unit_bytes + off, buf, bytes);
    bulk_commit();
    bulk_wait_read_all();   // the shared-memory source stays until the copy has read it
}

}  // namespace

int read_and_clear_status_state_copy(cudaStream_t s, int32_t *status)
{
    int host = 0, zero = 0;
    if (cudaMemcpyFromSymbolAsync(&host, g_state_copy_error, sizeof(int), 0,
                                  cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return KDA_ERR_CUDA;
    if (cudaMemcpyToSymbolAsync(g_state_copy_error, &zero, sizeof(int), 0,
                                cudaMemcpyHostToDevice, s) != cudaSuccess)
        return KDA_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return KDA_ERR_CUDA;
    *status = host;
    return KDA_OK;
}

int launch_state_copy(float *dst, const int64_t *dst_idx, int64_t n_dst, const float *src,
                      const int64_t *src_idx, int64_t n_src, int64_t n, int64_t unit_floats,
                      cudaStream_t stream)
{
    if (n == 0 || unit_floats == 0) return KDA_OK;
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const unsigned ys = (unsigned)(n < 65535 ? n : 65535);
    const int64_t unit_bytes = unit_floats * 4, chunks = (unit_bytes + kChunkBytes - 1) / kChunkBytes;
    if (unit_floats % 4 == 0 && n * chunks <= 0x7fffffffLL) {
        if (cudaFuncSetAttribute(state_copy_bulk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)kChunkBytes) != cudaSuccess)
            return KDA_ERR_CUDA;
        state_copy_bulk_kernel<<<(unsigned)(n * chunks), 32, kChunkBytes, stream>>>(
            reinterpret_cast<char *>(dst), dst_idx, n_dst, reinterpret_cast<const char *>(src), src_idx,
            n_src, unit_bytes, chunks);
    } else if (unit_floats % 4 == 0) {
        const int64_t vecs = unit_floats / 4;
        // enough blocks per slot that every SM is fully occupied (8 blocks of 256 threads)
        int64_t bx = (8LL * sms + ys - 1) / ys;
        const int64_t need = (vecs + 255) / 256;
        if (bx > need) bx = need;
        if (bx < 1) bx = 1;
        state_copy_kernel<float4><<<dim3((unsigned)bx, ys), 256, 0, stream>>>(
            reinterpret_cast<float4 *>(dst), dst_idx, n_dst, reinterpret_cast<const float4 *>(src),
            src_idx, n_src, n, vecs);
    } else {
        int64_t bx = (8LL * sms + ys - 1) / ys;
        const int64_t need = (unit_floats + 255) / 256;
        if (bx > need) bx = need;
        if (bx < 1) bx = 1;
        state_copy_kernel<float><<<dim3((unsigned)bx, ys), 256, 0, stream>>>(
            dst, dst_idx, n_dst, src, src_idx, n_src, n, unit_floats);
    }
    return cudaGetLastError() == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

}  // namespace kda
