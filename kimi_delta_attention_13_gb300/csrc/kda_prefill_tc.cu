// kda_prefill_tc.cu -- tensor-core chunked KDA prefill for sm_103a (bf16 inputs, fp32 state).
//
// Operation ("Kimi K3 im Detail", section "Sequenz-Mixing: KDA-Zustand und globale MLA"): per
// head S' = diag(exp(clamp(g_t,-5,0))) S_{t-1}, S_t = S' + beta_t k_t (v_t - S'^T k_t)^T,
// o_t = S_t^T q_t.  Prefill handles the tokens of a chunk in parallel and hands the state from
// chunk to chunk; the -5 log-decay floor keeps the cumulative decay of a 16-token tile >= -80,
// which lets both the diagonal and the off-diagonal tile products run as tensor-core matmuls
// (same section, second paragraph).  This kernel keeps that tile bound and advances the state by
// C = 32 tokens (two tiles) per step.
//
// Chunk algebra for one step (S0 = state at the step start, G_r = cumulative clamped log-decay
// from the step start through token r, b_r = exp(G_r), per key channel):
//   u_r = beta_r (v_r - S0^T (k_r b_r) - sum_{s<r} ((k_r b_r).(k_s / b_s)) u_s)
//     =>  U = T diag(beta) (V - K~ S0),  T = (I + A)^-1,  A[r][s] = beta_r (k_r b_r).(k_s / b_s), s<r
//   o_r = S0^T (q_r b_r) + sum_{s<=r} ((q_r b_r).(k_s / b_s)) u_s      (mask includes the diagonal)
//   S_C = diag(b_C) S0 + sum_s (k_s b_C / b_s) u_s^T
// With Wm = T diag(beta) K~ and Um = T diag(beta) V:  V_new = Um - Wm S0,  O = Q~ S0 + Aqk V_new.
// Every exponential is formed inside one 16-token tile or relative to a tile boundary, so each
// factor lies in [e^-80, e^80] (Gram blocks: left operand relative to its own tile start, right
// operand relative to the row tile's start).
//
// Work split: one CTA per (sequence, head), 384 threads:
//   warp 0       TMA producer: q, k, g, v tiles (32 tokens x 128, 128-byte swizzle) + beta
//   warp 1       TMEM owner and the single MMA-issuing thread (tcgen05.mma, kind::f16)
//   warps 4..7   chain: thread j <-> TMEM lane j <-> value channel j; fp32 state S^T in TMEM,
//                its bf16 copy in TMEM as the A operand of the state products; outputs
//   warps 8..11  prep: state-independent work of the next step (decay cumprods, scaled bf16
//                operands, Gram post-processing, the 32x32 unit-triangular solve, W and U)
// Accumulators and A operands live in TMEM (512 columns); B operands in shared memory.
//
// Precision: the max-error bound (2e-2 x RMS on outputs, 1e-2 on states) needs ~1e-3 relative
// accuracy on the largest elements.  The Gram products (q.k with e^+-80 scalings, where the dot
// product cancels) therefore run as kind::tf32 on fp32 operands, the state products as fp16
// (10-bit mantissa; all their operands are O(1) after the tile scalings), and only the W / U
// products, whose dominant terms are exact, as bf16.
#include <cudaTypedefs.h>

#include <mutex>

#include "kda_internal.cuh"
#include "sm100_ptx.cuh"

namespace kda {
namespace {

using namespace ptx;

constexpr int D = 128;        // d_k = d_v
constexpr int C = 32;         // tokens per chain step
constexpr int kThreads = 384;
constexpr uint64_t kTimeoutNs = 2000000000ull;   // bounded waits: 2 s

// shared memory map (bytes from a 1024-aligned base)
constexpr int kQStages = 2;                                // q, k, g ring (read by the prep step)
constexpr int kVStages = 3;                                // v ring (read by the U product)
constexpr uint32_t TILE_BYTES = 2 * C * 128;               // 64 channels x 32 rows x 2 halves
constexpr uint32_t QSTAGE_BYTES = 3 * TILE_BYTES;          // q, k, g
constexpr uint32_t OFF_QRING = 0;
constexpr uint32_t OFF_VRING = OFF_QRING + kQStages * QSTAGE_BYTES;
constexpr uint32_t OFF_MMA1B = OFF_VRING + kVStages * TILE_BYTES;  // [-W^T | Q~^T] fp16, x2
constexpr uint32_t OFF_KK = OFF_MMA1B + 2 * 16384;                   // [Kbar fp16 | K~ bf16], x2
constexpr uint32_t OFF_AB = OFF_KK + 2 * 16384;                      // [Aqk fp16 | Bt bf16] 64 rows, x2
// Gram operands, fp32 K-major (tf32 product), 4 regions of 32 channels each.  A has M = 128 rows
// of which 64 are real (32 k-rows, 32 q-rows): its regions are spaced 64 rows apart, so the 64
// unused rows of one region read the next region (or Gram B), and their results are ignored.
constexpr uint32_t GA_REGION = 64 * 128, GB_REGION = 48 * 128;
constexpr uint32_t OFF_GA = OFF_AB + 2 * 8192;                       // Gram A: 4 x 8 KB
constexpr uint32_t OFF_GB = OFF_GA + 4 * GA_REGION;                  // Gram B: 4 x 6 KB (N = 48)
constexpr uint32_t OFF_BC = OFF_GB + 4 * GB_REGION;                  // step decay b_C, x2
constexpr uint32_t OFF_BETA = OFF_BC + 2 * D * 4;                    // beta per v stage
constexpr uint32_t OFF_BARS = OFF_BETA + kVStages * C * 4;
constexpr uint32_t NUM_BARS = 24;
constexpr uint32_t OFF_MISC = OFF_BARS + NUM_BARS * 8;
constexpr uint32_t SMEM_BYTES = OFF_MISC + 64;
constexpr uint32_t SMEM_ALLOC = SMEM_BYTES + 1024;                   // alignment slack
// fp32 scratch of the triangular solve, placed in the Gram B buffer, which is dead between the
// completion of the Gram product and the next step's operand writes
constexpr uint32_t OFF_SA = OFF_GB;                                  // A (fp32) 32 x 33
constexpr uint32_t OFF_ST = OFF_SA + C * 33 * 4;                     // T (fp32) 32 x 33
constexpr uint32_t OFF_SX = OFF_ST + C * 33 * 4;                     // A10 T00, 16 x 17
static_assert(OFF_SX + 16 * 17 * 4 <= OFF_GB + 4 * GB_REGION, "solve scratch fits in the Gram B buffer");
static_assert(SMEM_ALLOC <= 232448, "shared memory per block");

// TMEM column map
constexpr uint32_t TM_S32 = 0;      // fp32 state S^T (lane j, column = key channel)
constexpr uint32_t TM_SBF = 128;    // bf16 copy, A operand (64 columns)
constexpr uint32_t TM_D1 = 192;     // 2 x 64: [U^T -> V_new^T | Y^T -> O^T]
constexpr uint32_t TM_VBF = 320;    // bf16 V_new^T, A operand (16 columns)
constexpr uint32_t TM_DG = 352;     // Gram (48 columns)
constexpr uint32_t TM_DW = 416;     // W^T (32 columns)
constexpr uint32_t TM_COLS = 512;

// instruction descriptors (M = 128 everywhere)
constexpr uint32_t I_GRAM = idesc_f32acc(128, 48, FMT_TF32, 0, 0);
constexpr uint32_t I_W = idesc_f32acc(128, 32, FMT_BF16, 0, 0);
constexpr uint32_t I_U = idesc_f32acc(128, 64, FMT_BF16, 1, 0);
constexpr uint32_t I_MMA1 = idesc_f32acc(128, 64, FMT_F16, 0, 1);
constexpr uint32_t I_MMA2 = idesc_f32acc(128, 32, FMT_F16, 0, 0);
constexpr uint32_t I_MMA3 = idesc_f32acc(128, 128, FMT_F16, 0, 0);

enum Bar {
    B_QFULL = 0,         // + q stage (2)
    B_QEMPTY = 2,        // + q stage (2)
    B_VFULL = 4,         // + v stage (3)
    B_VEMPTY = 7,        // + v stage (3)
    B_GRAM_OPS = 10, B_GRAM_DONE, B_WU_OPS, B_WU_DONE, B_MMA1_OPS, B_MMA1_DONE, B_VNEW, B_MMA3_DONE,
    B_STATE, B_D1FREE = 19 /* +buf (2) */, B_CHAIN_SYNC = 21, B_PREP_SYNC = 22, B_COUNT = 23
};
static_assert(B_COUNT <= (int)NUM_BARS, "barrier slots");

struct Misc {
    uint32_t tmem_base;
    int abort;
    int seq;
    int pad;
    long long start, end, first_ckpt;
};

__device__ int g_prefill_tc_error;  // sticky device error word of this translation unit

struct Params {
    const __nv_bfloat16 *beta;
    const int32_t *cu_seqlens;
    int n_seqs;
    int H;
    long long total_tokens;
    const float *init;
    void *out;
    float *final_state;
    int ckpt_stride;
    float *ckpts;
};

__device__ __forceinline__ void fail(Misc *misc)
{
    atomicExch(&g_prefill_tc_error, KDA_ERR_DEVICE_TIMEOUT);
    misc->abort = 1;
}

__device__ __forceinline__ bool wait_bar(uint64_t *bar, uint32_t parity, Misc *misc)
{
    if (mbar_wait(bar, parity, &misc->abort, kTimeoutNs)) return true;
    fail(misc);
    return false;
}

// Barrier among the 128 threads of one group, built on an mbarrier so that a member that gave
// up (timeout or abort) cannot leave the others blocked: every wait here is bounded too.
struct GroupSync {
    uint64_t *bar;
    uint32_t phase;
    __device__ __forceinline__ bool sync(Misc *misc)
    {
        mbar_arrive(bar);
        const bool ok = wait_bar(bar, phase, misc);
        phase ^= 1u;
        return ok;
    }
};

__device__ __forceinline__ float bf2f(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d)
{
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d)
                 : "memory");
}

// 8 consecutive bf16 values (one 16-byte chunk) from fp32
__device__ __forceinline__ void store_chunk(uint32_t addr, const float *v)
{
    st_shared_v4(addr, pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]), pack_bf16x2(v[4], v[5]),
                 pack_bf16x2(v[6], v[7]));
}

__device__ __forceinline__ void store_chunk_f16(uint32_t addr, const float *v)
{
    st_shared_v4(addr, pack_f16x2(v[0], v[1]), pack_f16x2(v[2], v[3]), pack_f16x2(v[4], v[5]),
                 pack_f16x2(v[6], v[7]));
}

// one fp32 value rounded to the nearest tf32 (10-bit mantissa), so the tf32 product sees a
// round-to-nearest operand whatever it does with the low mantissa bits
__device__ __forceinline__ void store_tf32(uint32_t addr, float x)
{
    uint32_t t;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(t) : "f"(x));
    asm volatile("st.shared.b32 [%0], %1;" ::"r"(addr), "r"(t) : "memory");
}

template <typename TO>
__device__ __forceinline__ void store_out(TO *p, float x);
template <>
__device__ __forceinline__ void store_out<float>(float *p, float x) { *p = x; }
template <>
__device__ __forceinline__ void store_out<__nv_bfloat16>(__nv_bfloat16 *p, float x) { *p = __float2bfloat16_rn(x); }

// The work item of this CTA: the (blockIdx / H)-th longest sequence (ties by index), head
// blockIdx % H, so that long chains start first.  For very large batches: natural order.
__device__ void select_item(const Params &p, Misc *misc)
{
    const int rank = (int)(blockIdx.x / p.H);
    if (threadIdx.x == 0) misc->seq = rank;
    __syncthreads();
    if (p.cu_seqlens && p.n_seqs > 1 && p.n_seqs <= 2048) {
        for (int s = threadIdx.x; s < p.n_seqs; s += blockDim.x) {
            const int ls = p.cu_seqlens[s + 1] - p.cu_seqlens[s];
            int r = 0;
            for (int s2 = 0; s2 < p.n_seqs; ++s2) {
                const int l2 = p.cu_seqlens[s2 + 1] - p.cu_seqlens[s2];
                r += (l2 > ls) || (l2 == ls && s2 < s);
            }
            if (r == rank) misc->seq = s;
        }
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        const int n = misc->seq;
        misc->start = p.cu_seqlens ? p.cu_seqlens[n] : 0;
        misc->end = p.cu_seqlens ? p.cu_seqlens[n + 1] : p.total_tokens;
        long long first = 0;
        if (p.ckpt_stride > 0 && p.cu_seqlens)
            for (int m = 0; m < n; ++m) first += (p.cu_seqlens[m + 1] - p.cu_seqlens[m]) / p.ckpt_stride;
        misc->first_ckpt = first;
        misc->abort = 0;
    }
}

// ------------------------------------------------------------------------------------------------
// chain group: thread j owns TMEM lane j = value channel j

template <typename TO>
__device__ void chain_role(const Params &p, uint8_t *smem, uint64_t *bars, Misc *misc, int h,
                           int nsteps)
{
    const int j = threadIdx.x - 128;
    const int wq = j >> 5;  // TMEM sub-partition of this warp
    // TMEM A operands: fp16 state copy (TM_SBF) and fp16 V_new^T (TM_VBF)
    const uint32_t tb = misc->tmem_base + ((uint32_t)(32 * wq) << 16);
    const int n = misc->seq;
    const long long start = misc->start, end = misc->end;
    const long long sbase = ((long long)n * p.H + h) * D * D;
    const float *bc_all = reinterpret_cast<const float *>(smem + OFF_BC);
    GroupSync gs{&bars[B_CHAIN_SYNC], 0};

    // initial state: S^T[j][c] = S[c][j]
    for (int c0 = 0; c0 < D; c0 += 32) {
        uint32_t r[32];
#pragma unroll
        for (int i = 0; i < 32; ++i)
            r[i] = __float_as_uint(p.init ? p.init[sbase + (long long)(c0 + i) * D + j] : 0.f);
        tmem_st32(tb + TM_S32 + c0, r);
        uint32_t rb[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) rb[i] = pack_f16x2(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1]));
        tmem_st16(tb + TM_SBF + c0 / 2, rb);
    }
    tmem_wait_st();
    tc_fence_before();
    if (!gs.sync(misc)) return;
    if (j == 0) mbar_arrive(&bars[B_STATE]);

    TO *out = reinterpret_cast<TO *>(p.out);
    for (int s = 0; s < nsteps && !misc->abort; ++s) {
        const int buf = s & 1;
        const uint32_t ph = s & 1;
        const long long t0 = start + (long long)s * C;
        const int valid = (int)((end - t0) < C ? (end - t0) : C);
        const float *bc = bc_all + buf * D;

        // decay the fp32 state by the step's b_C while MMA1 runs on the bf16 copy
        if (!wait_bar(&bars[B_MMA1_OPS], ph, misc)) break;
        for (int c0 = 0; c0 < D; c0 += 32) {
            uint32_t r[32];
            tmem_ld32(tb + TM_S32 + c0, r);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * bc[c0 + i]);
            tmem_st32(tb + TM_S32 + c0, r);
        }
        // V_new^T (fp32, from MMA1) -> fp16 A operand of the output and state products
        if (!wait_bar(&bars[B_MMA1_DONE], ph, misc)) break;
        tc_fence_after();
        {
            uint32_t r[32], rb[16];
            tmem_ld32(tb + TM_D1 + 64 * buf, r);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 16; ++i) rb[i] = pack_f16x2(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1]));
            tmem_st16(tb + TM_VBF, rb);
        }
        tmem_wait_st();
        tc_fence_before();
        if (!gs.sync(misc)) break;
        if (j == 0) mbar_arrive(&bars[B_VNEW]);

        // updated state: checkpoints / final state, bf16 copy for the next step
        if (!wait_bar(&bars[B_MMA3_DONE], ph, misc)) break;
        tc_fence_after();
        const long long done = (long long)(s + 1) * C;
        const bool last = (s == nsteps - 1);
        const bool ckpt = p.ckpt_stride > 0 && done <= end - start && (done % p.ckpt_stride) == 0;
        float *ck = nullptr;
        if (ckpt)
            ck = p.ckpts + ((misc->first_ckpt + done / p.ckpt_stride - 1) * p.H + h) * (long long)D * D;
        for (int c0 = 0; c0 < D; c0 += 32) {
            uint32_t r[32], rb[16];
            tmem_ld32(tb + TM_S32 + c0, r);
            tmem_wait_ld();
            if (ck) {
#pragma unroll
                for (int i = 0; i < 32; ++i) ck[(long long)(c0 + i) * D + j] = __uint_as_float(r[i]);
            }
            if (last && p.final_state) {
#pragma unroll
                for (int i = 0; i < 32; ++i) p.final_state[sbase + (long long)(c0 + i) * D + j] = __uint_as_float(r[i]);
            }
#pragma unroll
            for (int i = 0; i < 16; ++i) rb[i] = pack_f16x2(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1]));
            tmem_st16(tb + TM_SBF + c0 / 2, rb);
        }
        tmem_wait_st();
        tc_fence_before();
        if (!gs.sync(misc)) break;
        if (j == 0) mbar_arrive(&bars[B_STATE]);

        // outputs of this step: O^T[j][r]
        {
            uint32_t r[32];
            tmem_ld32(tb + TM_D1 + 64 * buf + 32, r);
            tmem_wait_ld();
            TO *o = out + (t0 * p.H + h) * (long long)D + j;
#pragma unroll
            for (int i = 0; i < 32; ++i)
                if (i < valid) store_out<TO>(o + (long long)i * p.H * D, __uint_as_float(r[i]));
        }
        tc_fence_before();
        if (!gs.sync(misc)) break;
        if (j == 0) mbar_arrive(&bars[B_D1FREE + buf]);
    }
}

// ------------------------------------------------------------------------------------------------
// prep group: thread p = key channel c for the elementwise work

__device__ void prep_role(const Params &p, uint8_t *smem, uint64_t *bars, Misc *misc, int nsteps)
{
    const int c = threadIdx.x - 256;           // key channel in the elementwise phase
    const int warp = c >> 5, lane = c & 31;    // warp 8 + warp; TMEM sub-partition = warp
    const uint32_t sbase = smem_u32(smem);
    const uint32_t tb = misc->tmem_base + ((uint32_t)(32 * warp) << 16);
    float *sA = reinterpret_cast<float *>(smem + OFF_SA);
    float *sT = reinterpret_cast<float *>(smem + OFF_ST);
    float *sX = reinterpret_cast<float *>(smem + OFF_SX);
    const float *sbeta_all = reinterpret_cast<const float *>(smem + OFF_BETA);
    float *bc_all = reinterpret_cast<float *>(smem + OFF_BC);
    const long long start = misc->start, end = misc->end;
    constexpr float LOG2E = 1.4426950408889634f;
    GroupSync gs{&bars[B_PREP_SYNC], 0};

    for (int s = 0; s < nsteps && !misc->abort; ++s) {
        const int qs = s % kQStages, vs = s % kVStages, buf = s & 1;
        const uint32_t ph = s & 1;
        const long long t0 = start + (long long)s * C;
        const int valid = (int)((end - t0) < C ? (end - t0) : C);
        const uint8_t *qkg = smem + OFF_QRING + qs * QSTAGE_BYTES;   // q, k, g tiles
        const float *sbeta = sbeta_all + vs * C;
        if (!wait_bar(&bars[B_QFULL + qs], (s / kQStages) & 1, misc)) break;

        // ---- P1: decay factors of channel c and the scaled operands --------------------------
        const uint32_t tile_off = (c >> 6) * 4096;
        float F[C], G[C];
        {
            float a[C];
#pragma unroll
            for (int r = 0; r < C; ++r) {
                const uint16_t gb = *reinterpret_cast<const uint16_t *>(qkg + 2 * TILE_BYTES + tile_off + sw128(r, (c & 63) * 2));
                float g = r < valid ? bf2f(gb) : 0.f;
                g = fminf(fmaxf(g, -5.0f), 0.0f);
                a[r] = exp2f(g * LOG2E);
            }
#pragma unroll
            for (int tile = 0; tile < 2; ++tile) {
                float f = 1.f;
#pragma unroll
                for (int r = 0; r < 16; ++r) { f *= a[16 * tile + r]; F[16 * tile + r] = f; }
                float gacc = 1.f;
#pragma unroll
                for (int r = 15; r >= 0; --r) { G[16 * tile + r] = gacc; gacc *= a[16 * tile + r]; }
            }
        }
        const float B0 = F[15], B1 = F[31];
        bc_all[buf * D + c] = B0 * B1;
        const uint32_t mma1b = sbase + OFF_MMA1B + buf * 16384;
        const uint32_t kk = sbase + OFF_KK + buf * 16384;
        const uint32_t ga_c = sbase + OFF_GA + (c >> 5) * GA_REGION;
        const uint32_t gb_c = sbase + OFF_GB + (c >> 5) * GB_REGION;
        const uint32_t cb = (c & 31) * 4;
#pragma unroll
        for (int m = 0; m < 4; ++m) {  // 8-token groups
            float kv[8], qv[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int r = 8 * m + i;
                const uint32_t off = tile_off + sw128(r, (c & 63) * 2);
                const bool ok = r < valid;
                qv[i] = ok ? bf2f(*reinterpret_cast<const uint16_t *>(qkg + off)) : 0.f;
                kv[i] = ok ? bf2f(*reinterpret_cast<const uint16_t *>(qkg + TILE_BYTES + off)) : 0.f;
            }
            float t[8];
            // E_r: decay from the step start through r (tile 1 adds tile 0's full decay)
#pragma unroll
            for (int i = 0; i < 8; ++i) t[i] = qv[i] * (m < 2 ? F[8 * m + i] : F[8 * m + i] * B0);
            store_chunk_f16(mma1b + sw128(c, (4 + m) * 16), t);             // Q~   (MMA1 B, N=32+r)
#pragma unroll
            for (int i = 0; i < 8; ++i) t[i] = kv[i] * (m < 2 ? F[8 * m + i] : F[8 * m + i] * B0);
            store_chunk(kk + sw128(c, (4 + m) * 16), t);                    // K~   (W A, bf16, k=s)
#pragma unroll
            for (int i = 0; i < 8; ++i) t[i] = kv[i] * (m < 2 ? G[8 * m + i] * B1 : G[8 * m + i]);
            store_chunk_f16(kk + sw128(c, m * 16), t);                      // Kbar (MMA3 B, k=r)
            // Gram operands, fp32 K-major (tf32 product): row = token (A: k rows 0..31, q rows
            // 32..63; B: k/F rows 0..31, tile-0 k*G rows 32..47), column = channel
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int r = 8 * m + i;
                store_tf32(ga_c + sw128(r, cb), kv[i] * F[r]);                      // K_L
                store_tf32(ga_c + sw128(32 + r, cb), qv[i] * F[r]);                 // Q_L
                store_tf32(gb_c + sw128(r, cb), kv[i] * __fdividef(1.f, F[r]));     // k / F
                if (m < 2) store_tf32(gb_c + sw128(32 + r, cb), kv[i] * G[r]);      // tile 0 rel. end
            }
        }
        fence_proxy_async_smem();
        if (!gs.sync(misc)) break;
        if (c == 0) {
            mbar_arrive(&bars[B_GRAM_OPS]);
            mbar_arrive(&bars[B_QEMPTY + qs]);   // q, k, g of this step fully read
        }

        // ---- P3: Gram -> A (fp32, beta folded) and Aqk (fp16 B operand) ----------------------
        if (!wait_bar(&bars[B_VFULL + vs], (s / kVStages) & 1, misc)) break;   // beta
        if (!wait_bar(&bars[B_GRAM_DONE], ph, misc)) break;
        tc_fence_after();
        if (warp < 2) {
            uint32_t r0[32], r1[16];
            tmem_ld32(tb + TM_DG, r0);
            tmem_ld16(tb + TM_DG + 32, r1);
            tmem_wait_ld();
            const int r = lane;   // token row
            // Gram(r, i): row tile 0 -> column i; row tile 1 -> column 32 + i for i in tile 0
            // (right operand relative to the end of tile 0), column i for i in tile 1.
            auto gram = [&](int i) -> float {
                return __uint_as_float((r >= 16 && i < 16) ? r1[i & 15] : r0[i & 31]);
            };
            if (warp == 0) {
                const float br = sbeta[r];
#pragma unroll
                for (int i = 0; i < C; ++i) sA[r * 33 + i] = (i < r) ? br * gram(i) : 0.f;
            } else {
                const uint32_t ab = sbase + OFF_AB + buf * 8192;
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    float t[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) t[i] = (8 * m + i <= r) ? gram(8 * m + i) : 0.f;
                    store_chunk_f16(ab + sw128(r, m * 16), t);              // Aqk row r (MMA2 B)
                }
            }
        }
        if (!gs.sync(misc)) break;

        // ---- P4: T = (I + A)^-1, blocked by 16x16 tiles ---------------------------------------
        if (warp == 0) {
            const int blk = lane >> 4, col = lane & 15, o = 16 * blk;
            float x[16];
#pragma unroll
            for (int r = 0; r < 16; ++r) {
                float acc = (r == col) ? 1.f : 0.f;
#pragma unroll
                for (int q = 0; q < r; ++q) acc -= sA[(o + r) * 33 + o + q] * x[q];
                x[r] = acc;
            }
#pragma unroll
            for (int r = 0; r < 16; ++r) sT[(o + r) * 33 + o + col] = x[r];
        }
        if (!gs.sync(misc)) break;
        for (int e = c; e < 256; e += 128) {    // X = A10 T00
            const int r = e >> 4, cc = e & 15;
            float acc = 0.f;
            for (int q = cc; q < 16; ++q) acc += sA[(16 + r) * 33 + q] * sT[q * 33 + cc];
            sX[r * 17 + cc] = acc;
        }
        if (!gs.sync(misc)) break;
        for (int e = c; e < 256; e += 128) {    // T10 = -T11 X
            const int r = e >> 4, cc = e & 15;
            float acc = 0.f;
            for (int q = 0; q <= r; ++q) acc += sT[(16 + r) * 33 + 16 + q] * sX[q * 17 + cc];
            sT[(16 + r) * 33 + cc] = -acc;
            sT[cc * 33 + 16 + r] = 0.f;          // upper block
        }
        if (!gs.sync(misc)) break;
        if (warp == 0) {   // Bt[r][s] = beta_s T[r][s] (B operand of the W and U products, bf16)
            const int r = lane;
            const uint32_t ab = sbase + OFF_AB + buf * 8192;
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                float t[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int q = 8 * m + i;
                    t[i] = (q <= r) ? sbeta[q] * sT[r * 33 + q] : 0.f;
                }
                store_chunk(ab + sw128(r, (4 + m) * 16), t);
            }
        }
        fence_proxy_async_smem();
        if (!gs.sync(misc)) break;
        if (c == 0) mbar_arrive(&bars[B_WU_OPS]);

        // ---- P6: -W (from W^T in TMEM) into the MMA1 B operand; release the v stage ------------
        if (!wait_bar(&bars[B_WU_DONE], ph, misc)) break;
        tc_fence_after();
        {
            uint32_t r[32];
            tmem_ld32(tb + TM_DW, r);
            tmem_wait_ld();
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                float t[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) t[i] = -__uint_as_float(r[8 * m + i]);
                store_chunk_f16(mma1b + sw128(c, m * 16), t);
            }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        if (!gs.sync(misc)) break;
        if (c == 0) {
            mbar_arrive(&bars[B_MMA1_OPS]);
            mbar_arrive(&bars[B_VEMPTY + vs]);
        }
    }
}

// ------------------------------------------------------------------------------------------------
// MMA issuer (one thread)

__device__ void mma_role(uint8_t *smem, uint64_t *bars, Misc *misc, int nsteps)
{
    const uint32_t sb = smem_u32(smem);
    const uint32_t tm = misc->tmem_base;
    int g = 0, w = 0, m1 = 0, m3 = 0;
    uint64_t last_progress = globaltimer_ns();
    while (m3 < nsteps) {
        if (misc->abort) break;
        bool progressed = false;
        // state products of step m3: MMA2 (outputs) and MMA3 (state)
        if (m3 < m1 && mbar_try_wait(&bars[B_VNEW], m3 & 1)) {
            tc_fence_after();
            const int buf = m3 & 1;
            for (int k = 0; k < 2; ++k)
                mma_ts(tm + TM_D1 + 64 * buf + 32, tm + TM_VBF + 8 * k,
                       smem_desc(sb + OFF_AB + buf * 8192 + 32 * k, 0, 1024), I_MMA2, 1);
            for (int k = 0; k < 2; ++k)
                mma_ts(tm + TM_S32, tm + TM_VBF + 8 * k,
                       smem_desc(sb + OFF_KK + buf * 16384 + 32 * k, 0, 1024), I_MMA3, 1);
            mma_commit(&bars[B_MMA3_DONE]);
            ++m3;
            progressed = true;
        }
        // state reads of step m1: V_new^T = U^T - S^T W^T, Y^T = S^T Q~^T
        if (m1 < w && m1 == m3 && mbar_try_wait(&bars[B_MMA1_OPS], m1 & 1) &&
            mbar_try_wait(&bars[B_STATE], m1 & 1)) {
            tc_fence_after();
            const int buf = m1 & 1;
            for (int k = 0; k < 8; ++k)
                mma_ts(tm + TM_D1 + 64 * buf, tm + TM_SBF + 8 * k,
                       smem_desc(sb + OFF_MMA1B + buf * 16384 + 2048 * k, 16384, 1024), I_MMA1, 1);
            mma_commit(&bars[B_MMA1_DONE]);
            ++m1;
            progressed = true;
        }
        // W and U of step w (needs the chain to have consumed step w-1's products and read
        // the outputs of step w-2 from this D1 buffer)
        if (w < g && w <= m3 && mbar_try_wait(&bars[B_WU_OPS], w & 1) &&
            (w < 2 || mbar_try_wait(&bars[B_D1FREE + (w & 1)], ((w >> 1) - 1) & 1)) &&
            mbar_try_wait(&bars[B_VFULL + w % kVStages], (w / kVStages) & 1)) {
            tc_fence_after();
            const int buf = w & 1, stage = w % kVStages;
            const uint32_t ab = sb + OFF_AB + buf * 8192 + 64;
            for (int k = 0; k < 2; ++k)
                mma_ss(tm + TM_DW, smem_desc(sb + OFF_KK + buf * 16384 + 64 + 32 * k, 0, 1024),
                       smem_desc(ab + 32 * k, 0, 1024), I_W, k > 0);
            const uint32_t vt = sb + OFF_VRING + stage * TILE_BYTES;
            for (int k = 0; k < 2; ++k)
                mma_ss(tm + TM_D1 + 64 * buf, smem_desc(vt + 2048 * k, 4096, 1024),
                       smem_desc(ab + 32 * k, 0, 1024), I_U, k > 0);
            mma_commit(&bars[B_WU_DONE]);
            ++w;
            progressed = true;
        }
        // Gram of step g
        if (g < nsteps && g <= w && mbar_try_wait(&bars[B_GRAM_OPS], g & 1)) {
            tc_fence_after();
            for (int k = 0; k < 16; ++k)   // tf32: K = 8 channels (32 bytes) per instruction
                mma_ss_tf32(tm + TM_DG,
                            smem_desc(sb + OFF_GA + (k >> 2) * GA_REGION + (k & 3) * 32, 0, 1024),
                            smem_desc(sb + OFF_GB + (k >> 2) * GB_REGION + (k & 3) * 32, 0, 1024),
                            I_GRAM, k > 0);
            mma_commit(&bars[B_GRAM_DONE]);
            ++g;
            progressed = true;
        }
        if (progressed) {
            last_progress = globaltimer_ns();
        } else if (globaltimer_ns() - last_progress > kTimeoutNs) {
            fail(misc);
            break;
        }
    }
}

// ------------------------------------------------------------------------------------------------
// TMA producer (warp 0)

__device__ void producer_role(const Params &p, const CUtensorMap *mq, const CUtensorMap *mk,
                              const CUtensorMap *mg, const CUtensorMap *mv, uint8_t *smem,
                              uint64_t *bars, Misc *misc, int h, int nsteps)
{
    const int lane = threadIdx.x & 31;
    const long long start = misc->start, end = misc->end;
    float *sbeta_all = reinterpret_cast<float *>(smem + OFF_BETA);
    int issued = 0;
    for (int s = 0; s < nsteps; ++s) {
        if (misc->abort) break;
        const int qs = s % kQStages, vs = s % kVStages;
        if (s >= kQStages && !wait_bar(&bars[B_QEMPTY + qs], ((s / kQStages) - 1) & 1, misc)) break;
        if (s >= kVStages && !wait_bar(&bars[B_VEMPTY + vs], ((s / kVStages) - 1) & 1, misc)) break;
        const long long t0 = start + (long long)s * C;
        uint8_t *qkg = smem + OFF_QRING + qs * QSTAGE_BYTES;
        uint8_t *vt = smem + OFF_VRING + vs * TILE_BYTES;
        if (lane == 0) {
            mbar_arrive_expect_tx(&bars[B_QFULL + qs], QSTAGE_BYTES);
            const CUtensorMap *maps[3] = {mq, mk, mg};
#pragma unroll
            for (int x = 0; x < 3; ++x)
#pragma unroll
                for (int half = 0; half < 2; ++half)
                    tma_load_3d(qkg + x * TILE_BYTES + half * 4096, maps[x], &bars[B_QFULL + qs],
                                half * 64, h, (int)t0);
            mbar_arrive_expect_tx(&bars[B_VFULL + vs], TILE_BYTES);
#pragma unroll
            for (int half = 0; half < 2; ++half)
                tma_load_3d(vt + half * 4096, mv, &bars[B_VFULL + vs], half * 64, h, (int)t0);
        }
        const long long t = t0 + lane;
        sbeta_all[vs * C + lane] = t < end ? __bfloat162float(p.beta[t * p.H + h]) : 0.f;
        mbar_arrive(&bars[B_VFULL + vs]);
        issued = s + 1;
    }
    // never leave the CTA with copies in flight
    for (int s = (issued > kQStages ? issued - kQStages : 0); s < issued; ++s)
        mbar_wait(&bars[B_QFULL + s % kQStages], (s / kQStages) & 1, &misc->abort, kTimeoutNs);
    for (int s = (issued > kVStages ? issued - kVStages : 0); s < issued; ++s)
        mbar_wait(&bars[B_VFULL + s % kVStages], (s / kVStages) & 1, &misc->abort, kTimeoutNs);
}

template <typename TO>
__global__ void __launch_bounds__(kThreads, 1)
prefill_tc_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
                  const __grid_constant__ CUtensorMap mg, const __grid_constant__ CUtensorMap mv,
                  const Params p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + OFF_BARS);
    Misc *misc = reinterpret_cast<Misc *>(smem + OFF_MISC);
    const int warp = threadIdx.x >> 5;
    const int h = blockIdx.x % p.H;

    select_item(p, misc);
    if (threadIdx.x == 0) {
        for (int s = 0; s < kQStages; ++s) {
            mbar_init(&bars[B_QFULL + s], 1);        // the expect_tx arrival
            mbar_init(&bars[B_QEMPTY + s], 1);
        }
        for (int s = 0; s < kVStages; ++s) {
            mbar_init(&bars[B_VFULL + s], 1 + 32);   // expect_tx arrival + one per lane (beta)
            mbar_init(&bars[B_VEMPTY + s], 1);
        }
        for (int b = B_GRAM_OPS; b < B_CHAIN_SYNC; ++b) mbar_init(&bars[b], 1);
        mbar_init(&bars[B_CHAIN_SYNC], 128);
        mbar_init(&bars[B_PREP_SYNC], 128);
        fence_barrier_init();
    }
    if (warp == 0) {
        tma_prefetch_desc(&mq); tma_prefetch_desc(&mk); tma_prefetch_desc(&mg); tma_prefetch_desc(&mv);
    }
    if (warp == 1) {
        tmem_alloc(&misc->tmem_base, TM_COLS);
        tmem_relinquish();
    }
    // zero rows 32..63 of both [Aqk | Bt] buffers (the N=64 U product reads them as zeros)
    for (int e = threadIdx.x; e < 2 * 32 * 32; e += kThreads) {
        const int b = e >> 10, rw = (e >> 5) & 31, word = e & 31;
        reinterpret_cast<uint32_t *>(smem + OFF_AB + b * 8192 + (32 + rw) * 128)[word] = 0u;
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    const long long len = misc->end - misc->start;
    const int nsteps = (int)((len + C - 1) / C);
    if (nsteps == 0) {
        // empty sequence: the final state is the initial one
        if (p.final_state) {
            const long long sbase = ((long long)misc->seq * p.H + h) * D * D;
            for (int e = threadIdx.x; e < D * D; e += kThreads)
                p.final_state[sbase + e] = p.init ? p.init[sbase + e] : 0.f;
        }
    } else if (warp == 0) {
        producer_role(p, &mq, &mk, &mg, &mv, smem, bars, misc, h, nsteps);
    } else if (warp == 1) {
        if ((threadIdx.x & 31) == 0) mma_role(smem, bars, misc, nsteps);
        __syncwarp();
    } else if (warp >= 4 && warp < 8) {
        chain_role<TO>(p, smem, bars, misc, h, nsteps);
    } else if (warp >= 8) {
        prep_role(p, smem, bars, misc, nsteps);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(misc->tmem_base, TM_COLS);
}

// ------------------------------------------------------------------------------------------------
// host side

PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
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

bool make_map(CUtensorMap *map, const void *base, int H, int64_t T)
{
    auto enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)T};
    cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)H * D * 2};
    cuuint32_t box[3] = {64, 1, (cuuint32_t)C}, es[3] = {1, 1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box,
               es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <typename TO>
int launch_typed(const CUtensorMap &mq, const CUtensorMap &mk, const CUtensorMap &mg,
                 const CUtensorMap &mv, const Params &p, int blocks, cudaStream_t stream)
{
    static std::once_flag once;
    static cudaError_t attr_rc = cudaSuccess;
    std::call_once(once, [] {
        attr_rc = cudaFuncSetAttribute(prefill_tc_kernel<TO>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       SMEM_ALLOC);
    });
    if (attr_rc != cudaSuccess) return KDA_ERR_CUDA;
    prefill_tc_kernel<TO><<<blocks, kThreads, SMEM_ALLOC, stream>>>(mq, mk, mg, mv, p);
    return cudaGetLastError() == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

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
    const int64_t blocks = (int64_t)n_seqs * n_heads;
    if (blocks == 0) return KDA_OK;
    if (blocks > 0x7fffffffLL) return KDA_ERR_INVALID_ARG;
    CUtensorMap mq, mk, mg, mv;
    if (!make_map(&mq, q, n_heads, total_tokens) || !make_map(&mk, k, n_heads, total_tokens) ||
        !make_map(&mg, g, n_heads, total_tokens) || !make_map(&mv, v, n_heads, total_tokens))
        return KDA_ERR_CUDA;
    Params p;
    p.beta = static_cast<const __nv_bfloat16 *>(beta);
    p.cu_seqlens = cu_seqlens;
    p.n_seqs = n_seqs;
    p.H = n_heads;
    p.total_tokens = total_tokens;
    p.init = init_state;
    p.out = out;
    p.final_state = final_state;
    p.ckpt_stride = ckpt_stride;
    p.ckpts = ckpts;
    if (out_dtype == KDA_BF16) return launch_typed<__nv_bfloat16>(mq, mk, mg, mv, p, (int)blocks, stream);
    return launch_typed<float>(mq, mk, mg, mv, p, (int)blocks, stream);
}

}  // namespace kda
