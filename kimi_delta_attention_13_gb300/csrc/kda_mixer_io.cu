// kda_mixer_io.cu -- the steps just around the KDA recurrence: the pre-mixer, which turns the q,
// k, v projections and the gate pre-activations into the recurrence's inputs, and the output gate.
//
// Page "Kimi K3 im Detail", section "Sequenz-Mixing: KDA-Zustand und globale MLA": a short
// convolution of width 4 for the KDA projections (first paragraph) and an input-dependent output
// gate acting on the KDA path's output (third paragraph).  The page gives neither formula; the
// readings implemented here are:
//   y_t = w0 x_(t-3) + w1 x_(t-2) + w2 x_(t-1) + w3 x_t     causal depthwise, per channel, no
//         activation; tokens before a sequence's start are its conv history (zeros or 3 rows)
//   q = y_q / max(||y_q||_2, eps),  k = y_k / max(||y_k||_2, eps)   per (token, head);  v = y_v
//   g = clamp(-softplus(a), -5, 0),  beta = 1 / (1 + exp(-b))
//   out = o / (1 + exp(-z))
//
// Every kernel here streams HBM once (the roofline is bytes / bandwidth): 16-byte vector loads
// and stores of 8 channels per thread, fp32 arithmetic.  The pre-mixer is two launches: the
// convolution of q, k and v, whose threads walk a 256-token chunk with a 3-token register window
// and keep the next 8 (bf16) or 4 (fp32) tokens' loads in flight (the chunk's first tokens read a
// 3-token halo that the neighbouring chunk, scheduled next to it, has just brought into L2); and
// the gates, elementwise at full occupancy (their exp/log chains kept the convolution's warps
// waiting when both shared a kernel), launched as a programmatic dependent of the convolution.
#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int kMixThreads = 128;   // 8 channels per thread: 1024 channels per block
constexpr int kMixTokens = 256;    // tokens per pre-mixer block (fewer block start-ups and halos)
// tokens each pre-mixer thread keeps in flight: 8 of bf16 (16 B each), 4 of fp32 (32 B each)
template <typename T>
constexpr int mix_depth() { return sizeof(T) == 2 ? 8 : 4; }

// 8 consecutive elements <-> 8 floats (16-byte bf16 vector, or two 16-byte fp32 vectors)
__device__ __forceinline__ void load8(const __nv_bfloat16 *p, float (&v)[8])
{
    const uint4 r = *reinterpret_cast<const uint4 *>(p);
    const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        v[2 * i] = __uint_as_float(w[i] << 16);
        v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}
__device__ __forceinline__ void load8(const float *p, float (&v)[8])
{
    const float4 a = *reinterpret_cast<const float4 *>(p), b = *reinterpret_cast<const float4 *>(p + 4);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}
__device__ __forceinline__ void store8(__nv_bfloat16 *p, const float (&v)[8])
{
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
        w[i] = *reinterpret_cast<const uint32_t *>(&h);
    }
    *reinterpret_cast<uint4 *>(p) = make_uint4(w[0], w[1], w[2], w[3]);
}
__device__ __forceinline__ void store8(float *p, const float (&v)[8])
{
    *reinterpret_cast<float4 *>(p) = make_float4(v[0], v[1], v[2], v[3]);
    *reinterpret_cast<float4 *>(p + 4) = make_float4(v[4], v[5], v[6], v[7]);
}

// 8 elements as loaded (packed bf16 stays packed until used): the prefetch ring's entries,
// unpacked as 4 channel pairs
template <typename T>
struct Raw8;
template <>
struct Raw8<__nv_bfloat16> {
    uint4 u;
    __device__ __forceinline__ void load(const __nv_bfloat16 *p) { u = *reinterpret_cast<const uint4 *>(p); }
    __device__ __forceinline__ void unpack(float2 (&v)[4]) const
    {
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) v[i] = make_float2(__uint_as_float(w[i] << 16), __uint_as_float(w[i] & 0xffff0000u));
    }
};
template <>
struct Raw8<float> {
    float4 a, b;
    __device__ __forceinline__ void load(const float *p)
    {
        a = *reinterpret_cast<const float4 *>(p);
        b = *reinterpret_cast<const float4 *>(p + 4);
    }
    __device__ __forceinline__ void unpack(float2 (&v)[4]) const
    {
        v[0] = make_float2(a.x, a.y); v[1] = make_float2(a.z, a.w);
        v[2] = make_float2(b.x, b.y); v[3] = make_float2(b.z, b.w);
    }
};

// packed fp32 pairs (one f32x2 instruction per pair)
__device__ __forceinline__ float2 pair_fma(float2 a, float2 b, float2 c)
{
    unsigned long long r, pa, pb, pc;
    asm("mov.b64 %0, {%1, %2};" : "=l"(pa) : "f"(a.x), "f"(a.y));
    asm("mov.b64 %0, {%1, %2};" : "=l"(pb) : "f"(b.x), "f"(b.y));
    asm("mov.b64 %0, {%1, %2};" : "=l"(pc) : "f"(c.x), "f"(c.y));
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(pa), "l"(pb), "l"(pc));
    float2 v;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(v.x), "=f"(v.y) : "l"(r));
    return v;
}
__device__ __forceinline__ float2 pair_mul(float2 a, float2 b)
{
    unsigned long long r, pa, pb;
    asm("mov.b64 %0, {%1, %2};" : "=l"(pa) : "f"(a.x), "f"(a.y));
    asm("mov.b64 %0, {%1, %2};" : "=l"(pb) : "f"(b.x), "f"(b.y));
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(pa), "l"(pb));
    float2 v;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(v.x), "=f"(v.y) : "l"(r));
    return v;
}
__device__ __forceinline__ void store8(__nv_bfloat16 *p, const float2 (&v)[4])
{
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const __nv_bfloat162 h = __floats2bfloat162_rn(v[i].x, v[i].y);
        w[i] = *reinterpret_cast<const uint32_t *>(&h);
    }
    *reinterpret_cast<uint4 *>(p) = make_uint4(w[0], w[1], w[2], w[3]);
}
__device__ __forceinline__ void store8(float *p, const float2 (&v)[4])
{
    *reinterpret_cast<float4 *>(p) = make_float4(v[0].x, v[0].y, v[1].x, v[1].y);
    *reinterpret_cast<float4 *>(p + 4) = make_float4(v[2].x, v[2].y, v[3].x, v[3].y);
}

__device__ __forceinline__ float sigmoid(float x) { return __fdividef(1.0f, 1.0f + __expf(-x)); }

// clamp(-softplus(a), -5, 0): softplus(a) >= 5 for a >= 4.9933, so larger a need no evaluation
__device__ __forceinline__ float decay_gate(float a)
{
    return a >= 5.0f ? -5.0f : fmaxf(-__logf(1.0f + __expf(a)), -5.0f);
}

struct PremixArgs {
    const void *x[3];      // xq, xk, xv  [T, H, d]
    const float *w;        // [3, H*d, 4]
    const void *hist;      // [N, 3, 3, H*d] or null
    const int32_t *cu;     // [N+1] or null (one sequence)
    int n_seqs;
    long long T;
    int H, d;
    float eps;
    void *y[3];            // q, k, v  [T, H, d]
};

// The short convolution.  blockIdx.x: kMixTokens-token chunk, blockIdx.y: 1024-channel block,
// blockIdx.z: 0 = q, 1 = k (both normalised), 2 = v.  Thread: 8 channels [col, col + 8) of one
// head.
template <typename T>
__global__ void __launch_bounds__(kMixThreads) premix_conv_kernel(const PremixArgs p)
{
    // the gates kernel launched after this one reads none of its outputs: it may start as soon
    // as every block of this grid has started
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    constexpr int kMixDepth = mix_depth<T>();
    const int xi = blockIdx.z;
    const bool norm = xi < 2;
    const long long HD = (long long)p.H * p.d;
    const long long col = 8ll * ((long long)blockIdx.y * kMixThreads + threadIdx.x);
    const bool active = col < HD;
    const long long t0 = (long long)blockIdx.x * kMixTokens;
    const long long t1 = min(t0 + kMixTokens, p.T);
    // pointers picked without indexing the parameter arrays (which would copy them to local memory)
    const T *x = static_cast<const T *>(xi == 0 ? p.x[0] : xi == 1 ? p.x[1] : p.x[2]);
    T *y = static_cast<T *>(xi == 0 ? p.y[0] : xi == 1 ? p.y[1] : p.y[2]);

    // the sequence holding t0: the last n with cu[n] <= t0 (then cu[n+1] > t0)
    int n = 0;
    long long start = 0, next = p.T;
    if (p.cu) {
        int lo = 0, hi = p.n_seqs - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (p.cu[mid] <= t0) lo = mid; else hi = mid - 1;
        }
        n = lo;
        start = p.cu[n];
        next = p.cu[n + 1];
    }

    // taps as channel pairs: wt[k][i] = (w[c][k], w[c+1][k]) for channels c = col + 2i
    float2 wt[4][4];
    if (active) {
        const float4 *wp = reinterpret_cast<const float4 *>(p.w + ((long long)xi * HD + col) * 4);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float4 e = wp[2 * i], o = wp[2 * i + 1];
            wt[0][i] = make_float2(e.x, o.x); wt[1][i] = make_float2(e.y, o.y);
            wt[2][i] = make_float2(e.z, o.z); wt[3][i] = make_float2(e.w, o.w);
        }
    }
    // history row r (0, 1, 2 = the 3rd, 2nd, 1st token before the start) of sequence `seq`
    auto hist_row = [&](int seq, int r, float2 (&v)[4]) {
        Raw8<T> raw;
        if (active && p.hist) {
            raw.load(static_cast<const T *>(p.hist) + (((long long)seq * 3 + xi) * 3 + r) * HD + col);
            raw.unpack(v);
        } else {
#pragma unroll
            for (int i = 0; i < 4; ++i) v[i] = make_float2(0.f, 0.f);
        }
    };
    auto input = [&](long long t, float2 (&v)[4]) {   // t in [start - 3, t0)
        if (t >= start) {
            Raw8<T> raw;
            if (active) {
                raw.load(x + t * HD + col);
                raw.unpack(v);
            }
        } else {
            hist_row(n, 3 - (int)(start - t), v);
        }
    };
    float2 w3[4] = {}, w2[4] = {}, w1[4] = {};
    input(t0 - 3, w3);
    input(t0 - 2, w2);
    input(t0 - 1, w1);

    // the next kMixDepth tokens' x are in flight while one token is computed
    Raw8<T> ring[kMixDepth];
#pragma unroll
    for (int j = 0; j < kMixDepth; ++j) {
        const long long t = t0 + j;
        if (active && t < t1) ring[j].load(x + t * HD + col);
    }

    const int group = p.d >> 3;   // threads per head (a power of two <= 32)
    for (long long tb = t0; tb < t1; tb += kMixDepth) {
#pragma unroll
        for (int j = 0; j < kMixDepth; ++j) {
            const long long t = tb + j;
            if (t >= t1) break;
            float2 cur[4];
            ring[j].unpack(cur);
            if (active && t + kMixDepth < t1) ring[j].load(x + (t + kMixDepth) * HD + col);
            if (t == next) {
                // a new sequence starts at t: its window is its own history
                do {
                    ++n;
                    start = p.cu[n];
                    next = p.cu[n + 1];
                } while (next <= t);
                hist_row(n, 0, w3);
                hist_row(n, 1, w2);
                hist_row(n, 2, w1);
            }
            float2 o[4];
            float2 ss2 = make_float2(0.f, 0.f);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                o[i] = pair_fma(wt[3][i], cur[i], pair_fma(wt[2][i], w1[i], pair_fma(wt[1][i], w2[i], pair_mul(wt[0][i], w3[i]))));
                ss2 = pair_fma(o[i], o[i], ss2);
                w3[i] = w2[i];
                w2[i] = w1[i];
                w1[i] = cur[i];
            }
            if (norm) {
                // per-head sum of squares over the head's `group` threads (aligned lane groups)
                float ss = ss2.x + ss2.y;
                for (int m = group >> 1; m >= 1; m >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, m);
                const float inv = rsqrtf(fmaxf(ss, p.eps * p.eps));   // 1 / max(||y||, eps)
#pragma unroll
                for (int i = 0; i < 4; ++i) o[i] = pair_mul(o[i], make_float2(inv, inv));
            }
            if (active) store8(y + t * HD + col, o);
        }
    }
}

// The gates: g = clamp(-softplus(a), -5, 0) over n8 groups of 8 elements, beta = sigmoid(b) over
// nb elements (grid-stride loops)
template <typename T>
__global__ void __launch_bounds__(256) premix_gates_kernel(const T *a, const T *b, T *g, T *beta,
                                                           long long n8, long long nb)
{
    const long long stride = (long long)gridDim.x * blockDim.x;
    const long long i0 = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    for (long long i = i0; i < n8; i += stride) {
        Raw8<T> raw;
        raw.load(a + 8 * i);
        float2 v[4];
        raw.unpack(v);
#pragma unroll
        for (int c = 0; c < 4; ++c) v[c] = make_float2(decay_gate(v[c].x), decay_gate(v[c].y));
        store8(g + 8 * i, v);
    }
    for (long long i = i0; i < nb; i += stride) store_as(beta + i, sigmoid(to_f32(b[i])));
}

// out = o * sigmoid(z) over n elements; 8 per thread and step of a grid-stride loop
template <typename TO, typename TZ, typename TY>
__global__ void __launch_bounds__(256) output_gate_kernel(const TO *o, const TZ *z, TY *out, long long n)
{
    const long long n8 = n >> 3;
    const long long stride = (long long)gridDim.x * blockDim.x;
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n8; i += stride) {
        float ov[8], zv[8];
        load8(o + 8 * i, ov);
        load8(z + 8 * i, zv);
#pragma unroll
        for (int c = 0; c < 8; ++c) ov[c] *= sigmoid(zv[c]);
        store8(out + 8 * i, ov);
    }
    if (blockIdx.x == 0 && threadIdx.x < (n & 7)) {
        const long long i = 8 * n8 + threadIdx.x;
        store_as(out + i, to_f32(o[i]) * sigmoid(to_f32(z[i])));
    }
}

int sm_count()
{
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 148;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 148;
    return sms;
}

// The gates after the convolution, as a programmatic dependent launch: their blocks fill the SMs
// that the convolution's last wave leaves idle.  Work later in the stream still waits for both.
template <typename T>
cudaError_t launch_gates(const void *a, const void *b, void *g, void *beta, long long n8, long long nb,
                         dim3 grid, cudaStream_t stream)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, premix_gates_kernel<T>, static_cast<const T *>(a),
                              static_cast<const T *>(b), static_cast<T *>(g), static_cast<T *>(beta),
                              n8, nb);
}

template <typename TO, typename TZ>
int launch_gate_out(const void *o, const void *z, void *out, int out_dtype, long long n,
                    dim3 grid, cudaStream_t stream)
{
    if (out_dtype == KDA_BF16)
        output_gate_kernel<TO, TZ, __nv_bfloat16><<<grid, 256, 0, stream>>>(
            static_cast<const TO *>(o), static_cast<const TZ *>(z), static_cast<__nv_bfloat16 *>(out), n);
    else
        output_gate_kernel<TO, TZ, float><<<grid, 256, 0, stream>>>(
            static_cast<const TO *>(o), static_cast<const TZ *>(z), static_cast<float *>(out), n);
    return KDA_OK;
}

}  // namespace

int launch_premix(const void *xq, const void *xk, const void *xv, const void *a, const void *b,
                  const float *w, const void *hist, const int32_t *cu_seqlens, int n_seqs,
                  long long total_tokens, int n_heads, int d, float eps, int dtype, void *q,
                  void *k, void *v, void *g, void *beta, cudaStream_t stream)
{
    if (total_tokens == 0) return KDA_OK;
    PremixArgs p;
    p.x[0] = xq; p.x[1] = xk; p.x[2] = xv;
    p.w = w; p.hist = hist;
    p.cu = n_seqs == 1 ? nullptr : cu_seqlens;
    p.n_seqs = n_seqs;
    p.T = total_tokens;
    p.H = n_heads; p.d = d; p.eps = eps;
    p.y[0] = q; p.y[1] = k; p.y[2] = v;
    const long long HD = (long long)n_heads * d;
    const dim3 grid((unsigned)((total_tokens + kMixTokens - 1) / kMixTokens),
                    (unsigned)((HD / 8 + kMixThreads - 1) / kMixThreads), 3);
    const long long n8 = total_tokens * HD / 8, nb = total_tokens * n_heads;
    const long long want = (n8 + 255) / 256, cap = 8ll * sm_count();
    const dim3 ggrid((unsigned)(want < cap ? want : cap));
    if (dtype == KDA_BF16) {
        premix_conv_kernel<__nv_bfloat16><<<grid, kMixThreads, 0, stream>>>(p);
        if (cudaGetLastError() != cudaSuccess ||
            launch_gates<__nv_bfloat16>(a, b, g, beta, n8, nb, ggrid, stream) != cudaSuccess)
            return KDA_ERR_CUDA;
    } else {
        premix_conv_kernel<float><<<grid, kMixThreads, 0, stream>>>(p);
        if (cudaGetLastError() != cudaSuccess ||
            launch_gates<float>(a, b, g, beta, n8, nb, ggrid, stream) != cudaSuccess)
            return KDA_ERR_CUDA;
    }
    return KDA_OK;
}

int launch_output_gate(const void *o, int o_dtype, const void *z, int z_dtype, void *out,
                       int out_dtype, long long n, cudaStream_t stream)
{
    if (n == 0) return KDA_OK;
    // enough 256-thread blocks for 8 resident per SM, fewer when n is small
    const long long want = (n / 8 + 255) / 256;
    const long long cap = 8ll * sm_count();
    const dim3 grid((unsigned)(want < 1 ? 1 : (want < cap ? want : cap)));
    if (o_dtype == KDA_BF16 && z_dtype == KDA_BF16)
        launch_gate_out<__nv_bfloat16, __nv_bfloat16>(o, z, out, out_dtype, n, grid, stream);
    else if (o_dtype == KDA_BF16)
        launch_gate_out<__nv_bfloat16, float>(o, z, out, out_dtype, n, grid, stream);
    else if (z_dtype == KDA_BF16)
        launch_gate_out<float, __nv_bfloat16>(o, z, out, out_dtype, n, grid, stream);
    else
        launch_gate_out<float, float>(o, z, out, out_dtype, n, grid, stream);
    return cudaGetLastError() == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

}  // namespace kda
