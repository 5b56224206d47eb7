// kda_decode.cu -- one-token KDA update, state read once and written back in place.
//
// Operation ("Kimi K3 im Detail", section "Sequenz-Mixing: KDA-Zustand und globale MLA"):
// the fixed-size recurrent state replaces a per-token cache, so generating one token is one
// step of the recurrence on each (sequence, head):
//     S' = diag(alpha) S,  r_k = S'^T k,  r_q = S'^T q,  u = beta (v - r_k),
//     S  <- S' + k u^T,    o = S^T q = r_q + (k.q) u.
// The 64 KB fp32 state of a head is the whole cost (HBM-bound, ~1 flop/byte): each block
// streams it once with 128-bit loads, keeps it in registers across the two reductions and
// stores it back with 128-bit stores.
//
// Block = 256 threads (8 warps) per (sequence, head).  Warp w holds key rows i = w + 8m,
// lane l holds value columns 4l..4l+3, so every warp load is one contiguous 512-byte row.
// Column sums over i: per-thread partials over its 16 rows, then a cross-warp pass in
// shared memory.
#include "kda_internal.cuh"
#include "sm100_ptx.cuh"

namespace kda {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxDk = 128;
constexpr int kMaxDv = 128;
constexpr int kRowsPerWarp = kMaxDk / kWarps;  // 16

template <typename T, typename TO>
__global__ void __launch_bounds__(kThreads, 2)
decode_kernel(const T *__restrict__ q, const T *__restrict__ k, const T *__restrict__ v,
              const T *__restrict__ g, const T *__restrict__ beta, float *__restrict__ state,
              TO *__restrict__ out, int dk, int dv)
{
    const int64_t nh = blockIdx.x;  // sequence * H + head
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    __shared__ float s_k[kMaxDk], s_q[kMaxDk], s_a[kMaxDk], s_v[kMaxDv];
    __shared__ float s_part[2][kWarps][kMaxDv];
    __shared__ float s_r[2][kMaxDv];
    __shared__ float s_kq;

    float *S = state + nh * (int64_t)dk * dv;
    const bool col_ok = 4 * lane < dv;

    // The state loads go out first: they are the bytes this kernel exists to move.
    float4 st[kRowsPerWarp];
#pragma unroll
    for (int m = 0; m < kRowsPerWarp; ++m) {
        const int i = warp + kWarps * m;
        if (col_ok && i < dk)
            st[m] = __ldcs(reinterpret_cast<const float4 *>(S + (int64_t)i * dv + 4 * lane));
        else
            st[m] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    if (tid < dk) {
        s_k[tid] = to_f32(k[nh * dk + tid]);
        s_q[tid] = to_f32(q[nh * dk + tid]);
        s_a[tid] = retention(to_f32(g[nh * dk + tid]));
    }
    if (tid < dv) s_v[tid] = to_f32(v[nh * dv + tid]);
    const float b = to_f32(beta[nh]);
    __syncthreads();

    if (warp == 0) {  // k . q, needed only for the output
        float acc = 0.f;
        for (int i = lane; i < dk; i += 32) acc += s_k[i] * s_q[i];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
        if (lane == 0) s_kq = acc;
    }

    // decay, then the two column sums S'^T k and S'^T q over this thread's rows
    float rk[4] = {0.f, 0.f, 0.f, 0.f}, rq[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int m = 0; m < kRowsPerWarp; ++m) {
        const int i = warp + kWarps * m;
        if (i < dk) {
            const float a = s_a[i], ki = s_k[i], qi = s_q[i];
            st[m].x *= a; st[m].y *= a; st[m].z *= a; st[m].w *= a;
            rk[0] += st[m].x * ki; rk[1] += st[m].y * ki; rk[2] += st[m].z * ki; rk[3] += st[m].w * ki;
            rq[0] += st[m].x * qi; rq[1] += st[m].y * qi; rq[2] += st[m].z * qi; rq[3] += st[m].w * qi;
        }
    }
    if (col_ok) {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            s_part[0][warp][4 * lane + c] = rk[c];
            s_part[1][warp][4 * lane + c] = rq[c];
        }
    }
    __syncthreads();
    {
        const int which = tid >> 7, j = tid & 127;  // 256 threads = 2 sums x 128 columns
        if (j < dv) {
            float acc = 0.f;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) acc += s_part[which][w][j];
            s_r[which][j] = acc;
        }
    }
    __syncthreads();
    if (!col_ok) return;

    float u[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) u[c] = b * (s_v[4 * lane + c] - s_r[0][4 * lane + c]);

    if (warp == 0) {
        const float kq = s_kq;
        TO *o = out + nh * dv + 4 * lane;
#pragma unroll
        for (int c = 0; c < 4; ++c) store_as(o + c, s_r[1][4 * lane + c] + kq * u[c]);
    }

    // delta-rule write, stored in place
#pragma unroll
    for (int m = 0; m < kRowsPerWarp; ++m) {
        const int i = warp + kWarps * m;
        if (i < dk) {
            const float ki = s_k[i];
            float4 s = st[m];
            s.x += ki * u[0]; s.y += ki * u[1]; s.z += ki * u[2]; s.w += ki * u[3];
            __stcs(reinterpret_cast<float4 *>(S + (int64_t)i * dv + 4 * lane), s);
        }
    }
}

// d_k = d_v = 128: the 64 KB state of a head is one contiguous block, so it moves by one bulk
// copy each way and is worked on in shared memory.  Registers stay few, three blocks share an SM
// and up to three states per SM are in flight.
constexpr uint32_t kStateBytes = 128 * 128 * 4;
constexpr long long kDecodeTimeout = 2000000000ll;   // SM cycles (~1 s): bounded waits

__device__ int g_decode_error;   // sticky device error word of this translation unit

template <typename T, typename TO>
__global__ void __launch_bounds__(kThreads)
decode_bulk_kernel(const T *__restrict__ q, const T *__restrict__ k, const T *__restrict__ v,
                   const T *__restrict__ g, const T *__restrict__ beta, float *__restrict__ state,
                   TO *__restrict__ out)
{
    using namespace ptx;
    extern __shared__ __align__(128) float sS[];   // S[i][j], 128 x 128, row = key channel
    __shared__ __align__(8) uint64_t bar;
    __shared__ float s_k[kMaxDk], s_q[kMaxDk], s_a[kMaxDk], s_v[kMaxDv];
    __shared__ float s_part[kWarps][kMaxDv];   // one sum's per-warp partials at a time (3 blocks/SM)
    __shared__ float s_r[2][kMaxDv];
    __shared__ float s_kq;
    __shared__ int s_zero;   // the abort flag of the waits: never set, they end by timeout only
    const int64_t nh = blockIdx.x;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    float *S = state + nh * (int64_t)kMaxDk * kMaxDv;
    if (tid == 0) {
        s_zero = 0;
        mbar_init(&bar, 1);
        fence_barrier_init();
    }
    __syncthreads();
    if (tid == 0) {   // the state goes out first: it is the bytes this kernel exists to move
        mbar_arrive_expect_tx(&bar, kStateBytes);
        bulk_load_1d(sS, S, kStateBytes, &bar);
    }
    if (tid < kMaxDk) {
        s_k[tid] = to_f32(k[nh * kMaxDk + tid]);
        s_q[tid] = to_f32(q[nh * kMaxDk + tid]);
        s_a[tid] = retention(to_f32(g[nh * kMaxDk + tid]));
        s_v[tid] = to_f32(v[nh * kMaxDv + tid]);
    }
    const float b = to_f32(beta[nh]);
    __syncthreads();
    if (warp == 0) {  // k . q, needed only for the output
        float acc = 0.f;
        for (int i = lane; i < kMaxDk; i += 32) acc += s_k[i] * s_q[i];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
        if (lane == 0) s_kq = acc;
    }
    const bool landed = mbar_wait(&bar, 0, &s_zero, kDecodeTimeout);
    if (!__syncthreads_and(landed)) {
        if (tid == 0) {
            atomicExch(&g_decode_error, KDA_ERR_DEVICE_TIMEOUT);
            mbar_wait(&bar, 0, &s_zero, kDecodeTimeout);   // no copy left in flight at exit
        }
        return;
    }
    // decay, then the two column sums S'^T k and S'^T q over this thread's rows i = warp + 8m
    const float4 *S4 = reinterpret_cast<const float4 *>(sS);
    float rk[4] = {0.f, 0.f, 0.f, 0.f}, rq[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
    for (int m = 0; m < kRowsPerWarp; ++m) {
        const int i = warp + kWarps * m;
        const float a = s_a[i], ki = s_k[i] * a, qi = s_q[i] * a;
        const float4 s = S4[i * 32 + lane];
        rk[0] += s.x * ki; rk[1] += s.y * ki; rk[2] += s.z * ki; rk[3] += s.w * ki;
        rq[0] += s.x * qi; rq[1] += s.y * qi; rq[2] += s.z * qi; rq[3] += s.w * qi;
    }
    // cross-warp sums through one 4 KB buffer: first S'^T k, then S'^T q
#pragma unroll
    for (int which = 0; which < 2; ++which) {
#pragma unroll
        for (int c = 0; c < 4; ++c) s_part[warp][4 * lane + c] = which ? rq[c] : rk[c];
        __syncthreads();
        if (tid < kMaxDv) {
            float acc = 0.f;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) acc += s_part[w][tid];
            s_r[which][tid] = acc;
        }
        __syncthreads();
    }
    float u[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) u[c] = b * (s_v[4 * lane + c] - s_r[0][4 * lane + c]);
    if (warp == 0) {
        const float kq = s_kq;
        TO *o = out + nh * kMaxDv + 4 * lane;
#pragma unroll
        for (int c = 0; c < 4; ++c) store_as(o + c, s_r[1][4 * lane + c] + kq * u[c]);
    }
    // S = S' + k u^T in place, then one bulk store back
    float4 *W4 = reinterpret_cast<float4 *>(sS);
#pragma unroll 4
    for (int m = 0; m < kRowsPerWarp; ++m) {
        const int i = warp + kWarps * m;
        const float a = s_a[i], ki = s_k[i];
        float4 s = W4[i * 32 + lane];
        s.x = fmaf(s.x, a, ki * u[0]); s.y = fmaf(s.y, a, ki * u[1]);
        s.z = fmaf(s.z, a, ki * u[2]); s.w = fmaf(s.w, a, ki * u[3]);
        W4[i * 32 + lane] = s;
    }
    fence_proxy_async_smem();
    __syncthreads();
    if (tid == 0) {
        bulk_store_1d(S, sS, kStateBytes);
        bulk_commit();
        bulk_wait_read_all();   // the shared-memory source stays until the copy has read it
    }
}

}  // namespace

int read_and_clear_status_decode(cudaStream_t s, int32_t *status)
{
    int host = 0, zero = 0;
    if (cudaMemcpyFromSymbolAsync(&host, g_decode_error, sizeof(int), 0, cudaMemcpyDeviceToHost, s) !=
            cudaSuccess ||
        cudaMemcpyToSymbolAsync(g_decode_error, &zero, sizeof(int), 0, cudaMemcpyHostToDevice, s) !=
            cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return KDA_ERR_CUDA;
    *status = host;
    return KDA_OK;
}

int launch_decode(const void *q, const void *k, const void *v, const void *g, const void *beta,
                  float *state, void *out, int n_seqs, int n_heads, int d_k, int d_v, int dtype,
                  int out_dtype, cudaStream_t stream)
{
    if (d_k < 1 || d_k > kMaxDk || d_v < 4 || d_v > kMaxDv || d_v % 4 != 0)
        return KDA_ERR_UNSUPPORTED_SHAPE;
    const int64_t blocks = (int64_t)n_seqs * n_heads;
    if (blocks == 0) return KDA_OK;
    if (blocks > 0x7fffffffLL) return KDA_ERR_INVALID_ARG;
    const bool bulk = d_k == kMaxDk && d_v == kMaxDv;
    bool attr_ok = true;
    auto go = [&](auto in_tag, auto out_tag) {
        using T = decltype(in_tag);
        using TO = decltype(out_tag);
        if (bulk) {
            attr_ok = cudaFuncSetAttribute(decode_bulk_kernel<T, TO>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)kStateBytes) == cudaSuccess;
            if (attr_ok)
                decode_bulk_kernel<T, TO><<<(unsigned)blocks, kThreads, kStateBytes, stream>>>(
                    (const T *)q, (const T *)k, (const T *)v, (const T *)g, (const T *)beta, state,
                    (TO *)out);
        } else {
            decode_kernel<T, TO><<<(unsigned)blocks, kThreads, 0, stream>>>(
                (const T *)q, (const T *)k, (const T *)v, (const T *)g, (const T *)beta, state,
                (TO *)out, d_k, d_v);
        }
    };
    if (dtype == KDA_BF16) {
        if (out_dtype == KDA_BF16) go(__nv_bfloat16{}, __nv_bfloat16{}); else go(__nv_bfloat16{}, float{});
    } else {
        if (out_dtype == KDA_BF16) go(float{}, __nv_bfloat16{}); else go(float{}, float{});
    }
    return (attr_ok && cudaGetLastError() == cudaSuccess) ? KDA_OK : KDA_ERR_CUDA;
}

}  // namespace kda
