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
//     =>  U_new = T diag(beta) (V - K~ S0),  T = (I + A)^-1,  A[r][s] = beta_r (k_r b_r).(k_s / b_s), s<r
//   o_r = S0^T (q_r b_r) + sum_{s<=r} ((q_r b_r).(k_s / b_s)) u_s      (mask includes the diagonal)
//   S_C = diag(b_C) S0 + sum_s (k_s b_C / b_s) u_s^T
// With Dl = V - K~ S0 and Bt = T diag(beta), every product that involves the state is
//   Dl = V - K~ S0,   O = Q~ S0 + P Dl  (P = Aqk Bt),   S_C = diag(b_C) S0 + R^T Dl  (R = Bt^T Kbar),
// so the state reads need only the scaled q and k of the step, and P and R, which do not depend on
// the state, are formed beside the chain.  The kernel carries -Dl, -P and -R (the identity of the V
// product is -I and the solver writes -Bt): the products are unchanged and no operand needs an
// explicit negation.
// Every decay factor that scales an operand spans at most one 16-token tile or is taken relative
// to a tile boundary, so each such factor lies within e^80 (Gram blocks: left operand relative to
// its own tile start, right operand relative to the row tile's start); factors <= 1 may underflow,
// which only drops terms below fp32 resolution.
//
// Work split: one CTA per (sequence, head), 512 threads.  tcgen05.mma issue costs the issuing
// thread tens of cycles per instruction, so the MMAs are spread over threads that would otherwise
// wait:
//   warp 0 lane 0  asynchronous issuer: TMA loads of q, k, g (one stage) and v (three stages; two
//                  in the precise build), the V products, the state reads and the P / R^T
//                  products, each as soon as its inputs are ready (the q, k, g load first: prep
//                  waits on it)
//   warp 1         TMEM allocation; the solve's diagonal blocks T00, T11 and half of T10
//   warp 2         issues the step's Gram product and reads -A out of it (with beta, loaded one
//                  step ahead)
//   warp 3         reads Aqk out of the Gram; the other half of T10.  Warps 1 and 3 write
//                  -Bt^T = -(T diag(beta))^T, the B operand of the P and R^T products
//   warps 4..7     chain: thread j <-> TMEM lane j <-> value channel j.  fp32 state S^T in TMEM
//                  (pre-multiplied by the step's decay), its fp16 copy in TMEM as the A operand
//                  of the state reads; copies P and R into their operand buffers, forms Dl,
//                  issues the output and state-update products; writes outputs (TMA store),
//                  checkpoints and the final state
//   warps 8..15    prep: decay cumprods and every scaled operand of a step, up to three steps
//                  ahead of the chain
// Accumulators and A operands live in TMEM (512 columns); B operands in shared memory.
//
// Precision: the max-error bound (2e-2 x RMS on outputs, 1e-2 on states) needs ~1e-3 relative
// accuracy on the largest elements.  The Gram products (q.k with e^+-80 scalings, where the dot
// product cancels) therefore run as kind::tf32 on fp32 operands, and every other product as fp16
// (10-bit mantissa; all their operands are O(1) after the tile scalings); V enters exactly
// (bf16 times an identity).
//
// Precise mode: this file is compiled a second time with KDA_PRECISE=1 (kda_prefill_tc_precise.cu)
// for kda_prefill_precise.  There warp 3 also writes the low part Aqk - fp16(Aqk) of the output
// product's A operand (exact in fp32, then rounded to fp16), and the P product accumulates
// Aqk_lo Bt onto fp16(Aqk) Bt in TMEM with two more MMAs, before P is rounded to fp16 once: the
// output error from the rounding of Aqk, the largest term, goes away.  The low parts take the
// unused lower half of the [-I | 0] constant's buffer (two slots) and one v stage (the third
// slot): the v ring is two deep in this mode.
#include <cuda_fp16.h>
#include <cudaTypedefs.h>

#include <mutex>

#ifndef KDA_PRECISE
#define KDA_PRECISE 0
#endif
#if KDA_PRECISE
#define KDA_TC_EXPORT(name) name##_precise
#else
#define KDA_TC_EXPORT(name) name
#endif

#include "kda_internal.cuh"
#include "sm100_ptx.cuh"

namespace kda {
namespace {

using namespace ptx;

constexpr int D = 128;        // d_k = d_v
constexpr int C = 32;         // tokens per chain step
constexpr int kThreads = 512;
constexpr long long kTimeout = 4000000000ll;     // bounded waits: 4e9 SM cycles (~2 s)

// shared memory map (bytes from a 1024-aligned base)
constexpr int kQStages = 1;                                // q, k, g stage (read by prep)
constexpr int kSlots = 3;                                  // depth of the prep -> chain buffers
constexpr int kVStages = KDA_PRECISE ? 2 : 3;              // v ring (read by the V product)
constexpr uint32_t TILE_BYTES = 2 * C * 128;               // 64 channels x 32 rows x 2 halves
constexpr uint32_t QSTAGE_BYTES = 3 * TILE_BYTES;          // q, k, g
constexpr uint32_t OFF_QRING = 0;
constexpr uint32_t OFF_VRING = OFF_QRING + kQStages * QSTAGE_BYTES;
// per slot (step mod 3): MMA1 B operand [K~ | Q~] fp16, rows = key channel, 64 tokens (MN-major)
constexpr uint32_t OFF_MMA1B = OFF_VRING + kVStages * TILE_BYTES;
// two buffers of 128-byte rows (row = key channel); slot k uses bytes 64*(k&1) .. +63 of buffer
// k>>1: Kbar fp16 (A of the R product), then R fp16 (B of the state update).  Bytes 64..127 of
// rows 0..63 of buffer 1 hold the constant [-I | 0] (B of the V product).
constexpr uint32_t OFF_KK = OFF_MMA1B + kSlots * 16384;
// per slot, rows = token (32 rows): bytes 0..63 Aqk fp16 (A of the P product), then P fp16 (B of
// the output product); bytes 64..127 Bt^T fp16 (B of the P and R products)
constexpr uint32_t AB_BYTES = 32 * 128;
constexpr uint32_t OFF_AB = OFF_KK + 2 * 16384;
// precise mode: the third slot's Aqk low part (32 rows of 128 bytes, bytes 0..63 used)
constexpr uint32_t OFF_ALO2 = OFF_AB + kSlots * AB_BYTES;
constexpr uint32_t ALO2_BYTES = KDA_PRECISE ? 32 * 128 : 0;
// Gram operands, fp32 K-major (tf32 product), 4 regions of 32 channels each.  A has M = 128 rows
// of which 64 are real (32 k-rows, 32 q-rows): each region's descriptor starts 64 rows before
// it, so the real rows land in TMEM lanes 64..127 (read by warps 2 and 3) and the 64 leading rows
// read the previous region (or the AB buffers), whose results are ignored.
constexpr uint32_t GA_REGION = 64 * 128, GB_REGION = 48 * 128;
constexpr uint32_t OFF_GA = OFF_ALO2 + ALO2_BYTES;                   // Gram A: 4 x 8 KB
constexpr uint32_t OFF_GB = OFF_GA + 4 * GA_REGION;                  // Gram B: 4 x 6 KB (N = 48)
constexpr uint32_t OFF_BC = OFF_GB + 4 * GB_REGION;                  // step decay b_C, per slot
constexpr uint32_t OFF_SA = OFF_BC + kSlots * D * 4;                 // A (fp32) 32 x 36
constexpr uint32_t OFF_TOT = OFF_SA + C * 36 * 4;                    // per-quarter decay totals
constexpr uint32_t OFF_TB = OFF_TOT + 4 * 64 * 8;                    // T00 | T11 blocks, x2
constexpr uint32_t OFF_BETA = OFF_TB + 2 * 2048;                     // beta per step parity
// output tile of a full step, [32 tokens][128 channels] of the output type, stored by one TMA
constexpr uint32_t OFF_OSTAGE = OFF_BETA + 3 * C * 4;
constexpr uint32_t OFF_BARS = OFF_OSTAGE + C * D * 4;
constexpr uint32_t NUM_BARS = 40;
constexpr uint32_t OFF_MISC = OFF_BARS + NUM_BARS * 8;
constexpr uint32_t SMEM_BYTES = OFF_MISC + 64;
constexpr uint32_t SMEM_ALLOC = SMEM_BYTES + 1024;                   // alignment slack
static_assert(SMEM_ALLOC <= 232448, "shared memory per block");
static_assert(OFF_GA >= GA_REGION, "the first Gram region's leading rows stay inside the buffer");
static_assert(OFF_OSTAGE % 128 == 0, "TMA store source alignment");
static_assert(OFF_MMA1B % 1024 == 0 && OFF_ALO2 % 1024 == 0, "128-byte swizzle atoms");

// byte offsets of a slot's buffers; Kbar / R addresses add the slot's half-row offset before the
// swizzle: kk_base(k) + sw128(row, kk_half(k) + byte)
__host__ __device__ constexpr uint32_t mma1b_off(int k) { return OFF_MMA1B + k * 16384; }
__host__ __device__ constexpr uint32_t kk_base(int k) { return OFF_KK + (k >> 1) * 16384; }
__host__ __device__ constexpr uint32_t kk_half(int k) { return (k & 1) * 64; }
__host__ __device__ constexpr uint32_t ab_off(int k) { return OFF_AB + k * AB_BYTES; }
constexpr int kEyeSlot = 3;   // the [-I | 0] constant sits where a fourth Kbar slot would be
// precise mode: where slot k's Aqk low part starts (rows of 128 bytes; add alo_half(k) to a byte
// offset before the swizzle).  Slots 0 and 1: rows 64..95 and 96..127 of the constant's half of
// the second Kbar buffer, which the constant (rows 0..63) leaves free; slot 2: its own region.
// As an M = 128 A operand each descriptor also reads the 96 rows after its slot (ignored lanes),
// all inside shared memory.
__host__ __device__ constexpr uint32_t alo_rows(int k)
{
    return k < 2 ? OFF_KK + 16384 + (64 + 32 * k) * 128 : OFF_ALO2;
}
__host__ __device__ constexpr uint32_t alo_half(int k) { return k < 2 ? 64 : 0; }
static_assert(kk_base(kEyeSlot) == OFF_KK + 16384 && kk_half(kEyeSlot) == 64, "low parts beside the constant");

// TMEM column map
constexpr uint32_t TM_S32 = 0;      // fp32 state S^T (lane j, column = key channel)
constexpr uint32_t TM_SBF = 128;    // fp16 copy, A operand (64 columns)
constexpr uint32_t TM_D1 = 192;     // 2 x 64: [V^T -> Dl^T | Y^T -> O^T]
constexpr uint32_t TM_VBF = 320;    // fp16 Dl^T, A operand (16 columns)
constexpr uint32_t TM_DG = 352;     // Gram, 2 x 48 columns (step parity)
constexpr uint32_t TM_DP = 448;     // P (lanes 0..31, 32 columns)
constexpr uint32_t TM_DR = 480;     // R^T (lane = key channel, 32 columns)
constexpr uint32_t TM_COLS = 512;

// instruction descriptors (M = 128 everywhere)
constexpr uint32_t I_GRAM = idesc_f32acc(128, 48, FMT_TF32, 0, 0);
constexpr uint32_t I_VI = idesc_f32acc(128, 64, FMT_BF16, 1, 0);
constexpr uint32_t I_PR = idesc_f32acc(128, 32, FMT_F16, 0, 0);
constexpr uint32_t I_MMA1 = idesc_f32acc(128, 64, FMT_F16, 0, 1);
constexpr uint32_t I_MMA2 = idesc_f32acc(128, 32, FMT_F16, 0, 0);
constexpr uint32_t I_MMA3 = idesc_f32acc(128, 128, FMT_F16, 0, 0);

// mbarriers.  A handoff that a group can run ahead of has one barrier per buffer slot, so that no
// waiter can ever be two phases behind the barrier it polls.
enum Bar {
    B_QFULL = 0,                 // TMA landed q, k, g
    B_QEMPTY = 1,                // prep read them
    B_VFULL = 2,                 // + v stage (3): TMA landed v
    B_VEMPTY = 5,                // + v stage (3): the V product of the step completed
    B_OPS_READY = 8,             // + slot (3): prep wrote the step's operands and b_C
    B_GRAM_DONE = 11,            // + step parity (2): Gram product complete
    B_EXTR_DONE = 13,            // + step parity (2): warps 2-3 read the Gram accumulator
    B_A_READY = 15,              // A and Aqk of the step are in shared memory
    B_SA_FREE = 16,              // the solver read A
    B_BT_READY = 17,             // + slot (3): Bt of the step is in shared memory
    B_PR_DONE = 20,              // P and R^T products complete
    B_MMA1_DONE = 21,            // state reads complete
    B_MMA3_DONE = 22,            // output and state-update products complete
    B_OPS_FREE = 23,             // + slot (3): every product of the step completed
    B_DRAIN = 26,                // + issuing thread (3): end-of-kernel drain of in-flight MMAs
    B_SBF_READY = 29,            // the chain wrote the fp16 state copy the next state read uses
    B_PR_FREE = 30,              // the chain read P and R^T out of TMEM
    B_D1_FREE = 31,              // + step parity (2): the chain read a step's outputs
    B_T_READY = 33,              // + step parity (2): phase 1 of the solve wrote T00 and T11
    B_GOPS_READY = 35,           // prep wrote the Gram operands of the step
    B_COUNT = 36
};
static_assert(B_COUNT <= (int)NUM_BARS, "barrier slots");

struct Misc {
    uint32_t tmem_base;
    int abort;
    int seq;
    int zero;          // always 0: the abort flag of waits that must not give up early
    long long start, end, first_ckpt;
};

__device__ int g_prefill_tc_error;  // sticky device error word of this translation unit
__device__ int g_prefill_tc_debug_site;   // the first failed bounds check (site number), 0 if none

// ---- bounds checks.  A build with -DKDA_DEBUG checks every shared-memory pointer the kernel's
// accessors take against the CTA's dynamic shared-memory window, and every TMEM address against
// the 512 allocated columns and the lanes the executing warp may reach (its 32-lane sub-partition);
// a failed check records KDA_ERR_DEVICE_BOUNDS and its site in device words and skips the access.
// Release builds compile the checks out.
extern __shared__ __align__(16) uint8_t kda_dyn_smem[];

__device__ __noinline__ void bounds_failed(int site)
{
    atomicCAS(&g_prefill_tc_debug_site, 0, site);
    atomicExch(&g_prefill_tc_error, KDA_ERR_DEVICE_BOUNDS);
}

__device__ __forceinline__ bool smem_in_window(const void *p, uint32_t bytes, int site)
{
    const uint32_t a = smem_u32(p), lo = smem_u32(kda_dyn_smem);
    if (a >= lo && a + bytes <= lo + SMEM_ALLOC) return true;
    bounds_failed(site);
    return false;
}

__device__ __forceinline__ bool tmem_in_reach(uint32_t taddr, uint32_t ncols, int site)
{
    const uint32_t lane = taddr >> 16, col = taddr & 0xffffu;
    if (lane == 32u * ((threadIdx.x >> 5) & 3u) && col + ncols <= 512u) return true;
    bounds_failed(site);
    return false;
}

#ifdef KDA_DEBUG
#define KDA_SMEM_OK(p, n, site) smem_in_window((p), (n), (site))
#define KDA_TMEM_OK(t, n, site) tmem_in_reach((t), (n), (site))
#else
#define KDA_SMEM_OK(p, n, site) true
#define KDA_TMEM_OK(t, n, site) true
#endif

// Per-step timeline of the first CTA (SM clock stamps), compiled in only with -DKDA_TRACE.
#ifdef KDA_TRACE
__device__ long long g_kda_trace[32 * 64];
#define KDA_TRACE_EVENT(ev, s)                                                        \
    do {                                                                              \
        if (blockIdx.x == 0 && (s) < 64) g_kda_trace[(ev) * 64 + (s)] = clock64();    \
    } while (0)
#else
#define KDA_TRACE_EVENT(ev, s) \
    do {                       \
    } while (0)
#endif

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

// Bounded wait; on failure the CTA's abort flag is raised and the caller carries on to its
// group's next vote, where the whole group leaves together.
__device__ __forceinline__ bool wait_bar(uint64_t *bar, uint32_t parity, Misc *misc)
{
    if (mbar_wait(bar, parity, &misc->abort, kTimeout)) return true;
    fail(misc);
    return false;
}

// Barrier among the `n` threads of one group (hardware barrier `id`).  It also votes on the
// CTA's abort flag, so the whole group takes the same decision to leave its loop: a member that
// gave up on a bounded wait never leaves the others blocked at a later barrier.
struct GroupSync {
    uint32_t id, n;
    __device__ __forceinline__ bool sync(Misc *misc) { return bar_and(id, n, misc->abort == 0); }
};

// Before the CTA exits (normally or after an abort), the thread that issued MMAs waits until
// they have all completed, so that no MMA still writes TMEM when it is released.
__device__ __forceinline__ void drain_mmas(uint64_t *bar, Misc *misc)
{
    mma_commit(bar);
    mbar_wait(bar, 0, &misc->zero, kTimeout);   // even after an abort: bounded by the timeout only
}

__device__ __forceinline__ void st_shared_v4(uint8_t *p, uint32_t a, uint32_t b, uint32_t c, uint32_t d)
{
    if (KDA_SMEM_OK(p, 16, 1)) *reinterpret_cast<uint4 *>(p) = make_uint4(a, b, c, d);
}

// TMEM loads and stores of this kernel (the warp-uniform address is checked in debug builds)
__device__ __forceinline__ void tld32(uint32_t t, uint32_t (&r)[32]) { if (KDA_TMEM_OK(t, 32, 2)) tmem_ld32(t, r); }
__device__ __forceinline__ void tld16(uint32_t t, uint32_t (&r)[16]) { if (KDA_TMEM_OK(t, 16, 3)) tmem_ld16(t, r); }
__device__ __forceinline__ void tst32(uint32_t t, const uint32_t (&r)[32]) { if (KDA_TMEM_OK(t, 32, 4)) tmem_st32(t, r); }
__device__ __forceinline__ void tst16(uint32_t t, const uint32_t (&r)[16]) { if (KDA_TMEM_OK(t, 16, 5)) tmem_st16(t, r); }

// 8 consecutive fp16 values (one 16-byte chunk) from fp32
__device__ __forceinline__ void store_chunk_f16(uint8_t *addr, const float *v)
{
    st_shared_v4(addr, pack_f16x2(v[0], v[1]), pack_f16x2(v[2], v[3]), pack_f16x2(v[4], v[5]),
                 pack_f16x2(v[6], v[7]));
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
        misc->zero = 0;
    }
}

// ------------------------------------------------------------------------------------------------
// packed fp32 pairs (two lanes of work per instruction)

__device__ __forceinline__ unsigned long long pk(float2 v)
{
    unsigned long long r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(v.x), "f"(v.y));
    return r;
}
__device__ __forceinline__ float2 upk(unsigned long long r)
{
    float2 v;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(v.x), "=f"(v.y) : "l"(r));
    return v;
}
__device__ __forceinline__ float2 mul2(float2 a, float2 b)
{
    unsigned long long r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(pk(a)), "l"(pk(b)));
    return upk(r);
}
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c)
{
    unsigned long long r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(pk(a)), "l"(pk(b)), "l"(pk(c)));
    return upk(r);
}

// ------------------------------------------------------------------------------------------------
// MMA issue (each called by one thread of the owning group)

// A shared-memory descriptor advanced by `bytes` (the start address is its low field, in 16-byte
// units; every operand here lies below 256 KB, so the field never carries)
__device__ __forceinline__ uint64_t desc_at(uint64_t d, uint32_t bytes) { return d + (bytes >> 4); }

// D1 of a step: [-V^T | 0] = V^T [-I | 0] (v tile as an MN-major A operand, exact in fp32)
__device__ __forceinline__ void issue_vi(uint32_t tm, uint32_t sb, int buf, int vs)
{
    const uint64_t a = smem_desc(sb + OFF_VRING + vs * TILE_BYTES, 4096, 1024);
    const uint64_t b = smem_desc(sb + kk_base(kEyeSlot) + kk_half(kEyeSlot), 0, 1024);
    const uint32_t d = tm + TM_D1 + 64 * buf;
    mma_ss(d, a, b, I_VI, 0);
    mma_ss(d, desc_at(a, 2048), desc_at(b, 32), I_VI, 1);
}

// state reads of a step: -Dl^T = -V^T + S^T K~^T (onto -V^T), Y^T = S^T Q~^T (onto zeros)
__device__ __forceinline__ void issue_mma1(uint32_t tm, uint32_t sb, int buf, int slot, uint64_t *done)
{
    const uint64_t b = smem_desc(sb + mma1b_off(slot), 16384, 1024);
    const uint32_t d = tm + TM_D1 + 64 * buf, a = tm + TM_SBF;
#pragma unroll
    for (int k = 0; k < 8; ++k) mma_ts(d, a + 8 * k, desc_at(b, 2048 * k), I_MMA1, 1);
    mma_commit(done);
}

// outputs O^T += Dl^T P^T and the state update S^T += Dl^T R
__device__ __forceinline__ void issue_mma23(uint32_t tm, uint32_t sb, int buf, int slot, uint64_t *done)
{
    const uint64_t bp = smem_desc(sb + ab_off(slot), 0, 1024);
    const uint64_t br = smem_desc(sb + kk_base(slot) + kk_half(slot), 0, 1024);
    const uint32_t a = tm + TM_VBF;
    mma_ts(tm + TM_D1 + 64 * buf + 32, a, bp, I_MMA2, 1);
    mma_ts(tm + TM_D1 + 64 * buf + 32, a + 8, desc_at(bp, 32), I_MMA2, 1);
    mma_ts(tm + TM_S32, a, br, I_MMA3, 1);
    mma_ts(tm + TM_S32, a + 8, desc_at(br, 32), I_MMA3, 1);
    mma_commit(done);
}

// Gram of a step (tf32: K = 8 channels, 32 bytes, per instruction); k-rows land in TMEM lanes
// 64..95, q-rows in lanes 96..127
__device__ __forceinline__ void issue_gram(uint32_t tm, uint32_t sb, int gb, uint64_t *done)
{
    const uint64_t a = smem_desc(sb + OFF_GA - GA_REGION, 0, 1024);
    const uint64_t b = smem_desc(sb + OFF_GB, 0, 1024);
#pragma unroll
    for (int k = 0; k < 16; ++k)
        mma_ss_tf32(tm + TM_DG + 48 * gb, desc_at(a, (k >> 2) * GA_REGION + (k & 3) * 32),
                    desc_at(b, (k >> 2) * GB_REGION + (k & 3) * 32), I_GRAM, k > 0);
    mma_commit(done);
}

// P = Aqk Bt (rows 0..31 of the A operand are Aqk: lanes 0..31) and R^T = Kbar^T Bt (lane = key
// channel); both with B = Bt^T rows
__device__ __forceinline__ void issue_pr(uint32_t tm, uint32_t sb, int slot, uint64_t *done)
{
    const uint64_t ab = smem_desc(sb + ab_off(slot), 0, 1024);
    const uint64_t kk = smem_desc(sb + kk_base(slot) + kk_half(slot), 0, 1024);
    const uint64_t bt = desc_at(ab, 64);
    mma_ss(tm + TM_DP, ab, bt, I_PR, 0);
    mma_ss(tm + TM_DP, desc_at(ab, 32), desc_at(bt, 32), I_PR, 1);
#if KDA_PRECISE
    const uint64_t lo = smem_desc(sb + alo_rows(slot) + alo_half(slot), 0, 1024);   // + Aqk_lo Bt
    mma_ss(tm + TM_DP, lo, bt, I_PR, 1);
    mma_ss(tm + TM_DP, desc_at(lo, 32), desc_at(bt, 32), I_PR, 1);
#endif
    mma_ss(tm + TM_DR, kk, bt, I_PR, 0);
    mma_ss(tm + TM_DR, desc_at(kk, 32), desc_at(bt, 32), I_PR, 1);
    mma_commit(done);
}

// ------------------------------------------------------------------------------------------------
// chain group: thread j owns TMEM lane j = value channel j

template <typename TO>
__device__ void chain_role(const Params &p, const CUtensorMap *mo, uint8_t *smem, uint64_t *bars,
                           Misc *misc, int h, int nsteps)
{
    const int j = threadIdx.x - 128;
    const int wq = j >> 5;  // TMEM sub-partition of this warp
    const uint32_t tm = misc->tmem_base;
    const uint32_t tb = tm + ((uint32_t)(32 * wq) << 16);
    const uint32_t sb = smem_u32(smem);
    const int n = misc->seq;
    const long long start = misc->start, end = misc->end;
    const long long sbase = ((long long)n * p.H + h) * D * D;
    const float *bc_all = reinterpret_cast<const float *>(smem + OFF_BC);
    GroupSync gs{1, 128};

    // initial state S^T[j][c] = S[c][j]: fp16 copy, and the fp32 state times step 0's decay
    wait_bar(&bars[B_OPS_READY + 0], 0, misc);
    for (int c0 = 0; c0 < D; c0 += 32) {
        uint32_t r[32], rb[16];
#pragma unroll
        for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(p.init ? p.init[sbase + (long long)(c0 + i) * D + j] : 0.f);
#pragma unroll
        for (int i = 0; i < 16; ++i) rb[i] = pack_f16x2(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1]));
        tst16(tb + TM_SBF + c0 / 2, rb);
#pragma unroll
        for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * bc_all[c0 + i]);
        tst32(tb + TM_S32 + c0, r);
    }
    tmem_wait_st();
    tc_fence_before();
    if (!gs.sync(misc)) return;
    if (j == 0) mbar_arrive(&bars[B_SBF_READY]);   // the first state read may go

    TO *out = reinterpret_cast<TO *>(p.out);
    for (int s = 0; s < nsteps; ++s) {
        const int buf = s & 1, vs = s % kVStages, slot = s % kSlots, nslot = (s + 1) % kSlots;
        const uint32_t ph = s & 1;
        const long long t0 = start + (long long)s * C;
        const int valid = (int)((end - t0) < C ? (end - t0) : C);
        const bool last = (s == nsteps - 1);

        // while the state reads run: R (all lanes) and P (lanes 0..31) into their operand buffers
        wait_bar(&bars[B_PR_DONE], ph, misc);
        if (j == 0) KDA_TRACE_EVENT(9, s);
        tc_fence_after();
        {
            uint32_t r[32];
            float t[8];
            tld32(tb + TM_DR, r);
            tmem_wait_ld();
            uint8_t *kk = smem + kk_base(slot);
#pragma unroll
            for (int m = 0; m < 4; ++m) {
#pragma unroll
                for (int i = 0; i < 8; ++i) t[i] = __uint_as_float(r[8 * m + i]);
                store_chunk_f16(kk + sw128(j, kk_half(slot) + 16 * m), t);   // R row = key channel j
            }
            if (wq == 0) {
                tld32(tb + TM_DP, r);
                tmem_wait_ld();
                uint8_t *ab = smem + ab_off(slot);
#pragma unroll
                for (int m = 0; m < 4; ++m) {
#pragma unroll
                    for (int i = 0; i < 8; ++i) t[i] = __uint_as_float(r[8 * m + i]);
                    store_chunk_f16(ab + sw128(j, 16 * m), t);        // P row = token j
                }
            }
            fence_proxy_async_smem();
            if (j == 0) KDA_TRACE_EVENT(10, s);
        }
        // Dl^T (fp32, from the state reads) -> fp16 A operand of the output and state products
        wait_bar(&bars[B_MMA1_DONE], ph, misc);
        if (j == 0) KDA_TRACE_EVENT(11, s);
        tc_fence_after();
        {
            uint32_t r[32], rb[16];
            tld32(tb + TM_D1 + 64 * buf, r);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 16; ++i) rb[i] = pack_f16x2(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1]));
            tst16(tb + TM_VBF, rb);
        }
        tmem_wait_st();
        tc_fence_before();
        if (!gs.sync(misc)) break;
        if (j == 0) {
            mbar_arrive(&bars[B_PR_FREE]);         // P and R^T read: the next ones may be issued
            mbar_arrive(&bars[B_VEMPTY + vs]);     // the V product of this step has completed
            tc_fence_after();
            issue_mma23(tm, sb, buf, slot, &bars[B_MMA3_DONE]);
            KDA_TRACE_EVENT(12, s);
        }

        // updated state S_{s+1}: checkpoint / final state and the fp16 copy for the next state
        // read first, so that the read is issued early; then the fp32 state pre-multiplied by
        // the next step's decay (needed only by the next state update)
        wait_bar(&bars[B_MMA3_DONE], ph, misc);
        tc_fence_after();
        if (j == 0) KDA_TRACE_EVENT(13, s);
        if (j == 0) mbar_arrive(&bars[B_OPS_FREE + slot]);   // this step's operand buffers are free
        const long long done = (long long)(s + 1) * C;
        const bool ckpt = p.ckpt_stride > 0 && done <= end - start && (done % p.ckpt_stride) == 0;
        float *ck = nullptr;
        if (ckpt)
            ck = p.ckpts + ((misc->first_ckpt + done / p.ckpt_stride - 1) * p.H + h) * (long long)D * D;
#pragma unroll 1
        for (int c0 = 0; c0 < D; c0 += 32) {
            uint32_t r[32], rb[16];
            tld32(tb + TM_S32 + c0, r);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 16; ++i) rb[i] = pack_f16x2(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1]));
            tst16(tb + TM_SBF + c0 / 2, rb);
            if (ck) {
#pragma unroll
                for (int i = 0; i < 32; ++i) ck[(long long)(c0 + i) * D + j] = __uint_as_float(r[i]);
            }
            if (last && p.final_state) {
#pragma unroll
                for (int i = 0; i < 32; ++i) p.final_state[sbase + (long long)(c0 + i) * D + j] = __uint_as_float(r[i]);
            }
        }
        if (j == 0) {
            KDA_TRACE_EVENT(14, s);
            bulk_wait_read_all();   // the previous output tile has left the staging buffer
        }
        tmem_wait_st();
        tc_fence_before();
        if (!gs.sync(misc)) break;
        if (j == 0) KDA_TRACE_EVENT(15, s);
        if (!last && j == 0) mbar_arrive(&bars[B_SBF_READY]);   // the next state read may go
        // outputs of this step: O^T[j][r].  A full step goes through the staging tile and one TMA
        // store; a ragged last step (whose box would reach into the next sequence) is stored
        // directly.
        {
            uint32_t r[32];
            tld32(tb + TM_D1 + 64 * buf + 32, r);
            tmem_wait_ld();
            if (valid == C && KDA_SMEM_OK(reinterpret_cast<TO *>(smem + OFF_OSTAGE) + j, (31 * D + 1) * sizeof(TO), 17)) {
                TO *st = reinterpret_cast<TO *>(smem + OFF_OSTAGE) + j;
#pragma unroll
                for (int i = 0; i < 32; ++i) store_out<TO>(st + i * D, __uint_as_float(r[i]));
                fence_proxy_async_smem();
            } else {
                TO *o = out + (t0 * p.H + h) * (long long)D + j;
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    if (i < valid) store_out<TO>(o + (long long)i * p.H * D, __uint_as_float(r[i]));
            }
        }
        tc_fence_before();
        if (!gs.sync(misc)) break;
        if (j == 0) {
            KDA_TRACE_EVENT(16, s);
            mbar_arrive(&bars[B_D1_FREE + buf]);   // outputs read: the V product two steps ahead
            if (valid == C) {
                tma_store_3d(mo, smem + OFF_OSTAGE, 0, h, (int)t0);
                bulk_commit();
            }
        }
        if (!last) {
            wait_bar(&bars[B_OPS_READY + nslot], ((s + 1) / kSlots) & 1, misc);   // b_C(s+1)
            const float *bcn = bc_all + nslot * D;
            if (!KDA_SMEM_OK(bcn, D * 4, 18)) bcn = bc_all;   // (debug: record, read in range)
#pragma unroll 1
            for (int c0 = 0; c0 < D; c0 += 32) {
                uint32_t r[32];
                tld32(tb + TM_S32 + c0, r);
                tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < 32; i += 4) {
                    const float4 b4 = *reinterpret_cast<const float4 *>(bcn + c0 + i);
                    const float2 lo = mul2(make_float2(__uint_as_float(r[i]), __uint_as_float(r[i + 1])), make_float2(b4.x, b4.y));
                    const float2 hi = mul2(make_float2(__uint_as_float(r[i + 2]), __uint_as_float(r[i + 3])), make_float2(b4.z, b4.w));
                    r[i] = __float_as_uint(lo.x); r[i + 1] = __float_as_uint(lo.y);
                    r[i + 2] = __float_as_uint(hi.x); r[i + 3] = __float_as_uint(hi.y);
                }
                tst32(tb + TM_S32 + c0, r);
            }
        }
        if (j == 0) KDA_TRACE_EVENT(17, s);

    }
    if (j == 0) {
        drain_mmas(&bars[B_DRAIN + 0], misc);
        bulk_wait_all();   // the last output tiles are written before the CTA leaves
    }
}

// ------------------------------------------------------------------------------------------------
// prep group (256 threads)

// 2^x for x in [-7.3, 0] (no denormal results): the hardware approximation, relative error
// below 2^-22
__device__ __forceinline__ float ex2_approx(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float2 bf2x2(uint32_t w)
{
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}

// Two fp32 values rounded half away from zero to tf32 (10-bit mantissa) by one 64-bit add of
// half a tf32 ulp to each bit pattern (no carry crosses the halves for finite values; the tf32
// product ignores the low 13 bits), so the Gram sees round-to-nearest operands.
__device__ __forceinline__ void store_tf32x2(uint8_t *addr, float2 v)
{
    if (KDA_SMEM_OK(addr, 8, 6)) *reinterpret_cast<unsigned long long *>(addr) = pk(v) + 0x0000100000001000ull;
}

// Decay factors and every scaled operand of step s.  Thread p owns the channel pair (2cp, 2cp+1)
// (x and y of every float2 below) and the 8 tokens of quarter qr (8qr .. 8qr+7; tile = qr / 2).
//   F = cumulative retention from the own tile's start through the token,
//   G = retention after the token through the own tile's end,
//   E = from the step's start through the token,  X = after the token through the step's end.
__device__ __forceinline__ void prep_operands(uint8_t *smem, const uint8_t *qkg, int p, int slot,
                                              int valid, Misc *misc, GroupSync &gs, bool &ok,
                                              uint64_t *bars, uint64_t *q_empty, int s)
{
    constexpr float LOG2E = 1.4426950408889634f;
    const int cp = p & 63, qr = p >> 6, tile = qr >> 1;
    const int c0 = 2 * cp;
    const uint32_t tile_off = (c0 >> 6) * 4096, cbyte = (c0 & 63) * 2;
    float2 *tot = reinterpret_cast<float2 *>(smem + OFF_TOT);
    float2 f[8], gl[8], kv[8], qv[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int r = 8 * qr + i;
        const uint32_t off = tile_off + sw128(r, cbyte);
        const bool in = r < valid && KDA_SMEM_OK(qkg + off, 2 * TILE_BYTES + 4, 7);
        const float2 g = in ? bf2x2(*reinterpret_cast<const uint32_t *>(qkg + 2 * TILE_BYTES + off)) : make_float2(0.f, 0.f);
        kv[i] = in ? bf2x2(*reinterpret_cast<const uint32_t *>(qkg + TILE_BYTES + off)) : make_float2(0.f, 0.f);
        qv[i] = in ? bf2x2(*reinterpret_cast<const uint32_t *>(qkg + off)) : make_float2(0.f, 0.f);
        const float2 gc = mul2(make_float2(fminf(fmaxf(g.x, -5.0f), 0.0f), fminf(fmaxf(g.y, -5.0f), 0.0f)),
                               make_float2(LOG2E, LOG2E));
        f[i] = make_float2(ex2_approx(gc.x), ex2_approx(gc.y));
    }
    // this warp holds its part of q, k, g in registers: release the stage (one arrival per warp)
    __syncwarp();
    if ((p & 31) == 0) mbar_arrive(q_empty);
    // quarter-local products: gl = after the token to the quarter end, f = through the token
    {
        float2 acc = make_float2(1.f, 1.f);
#pragma unroll
        for (int i = 7; i >= 0; --i) { gl[i] = acc; acc = mul2(acc, f[i]); }
#pragma unroll
        for (int i = 1; i < 8; ++i) f[i] = mul2(f[i], f[i - 1]);
    }
    if (KDA_SMEM_OK(tot + qr * 64 + cp, 8, 8)) tot[qr * 64 + cp] = f[7];
    ok = gs.sync(misc) && ok;
    // the previous Gram has read its operands
    if (s >= 1) wait_bar(&bars[B_GRAM_DONE + ((s - 1) & 1)], ((s - 1) >> 1) & 1, misc);
    if (p == 0) KDA_TRACE_EVENT(1, s);
    const float2 P0 = tot[cp], P1 = tot[64 + cp], P2 = tot[128 + cp], P3 = tot[192 + cp];
    const float2 B0 = mul2(P0, P1), B1 = mul2(P2, P3);
    const float2 one = make_float2(1.f, 1.f);
    const float2 pre = (qr & 1) ? (qr == 1 ? P0 : P2) : one;
    const float2 suf = (qr & 1) ? one : (qr == 0 ? P1 : P3);
    if (qr == 0 && KDA_SMEM_OK(smem + OFF_BC + slot * D * 4 + 8 * cp, 8, 9))
        reinterpret_cast<float2 *>(smem + OFF_BC + slot * D * 4)[cp] = mul2(B0, B1);
    const float2 emul = tile ? mul2(pre, B0) : pre;      // E = f * emul
    const float2 xmul = tile ? suf : mul2(suf, B1);      // X = gl * xmul
    // 1/F = G / (tile total): F G is the tile's total retention for every token of the tile, so
    // one reciprocal per channel replaces one per token (the total is >= e^-80, a normal float)
    const float2 Bt = tile ? B1 : B0;
    const float2 ginv = mul2(suf, make_float2(__fdividef(1.f, Bt.x), __fdividef(1.f, Bt.y)));
    uint8_t *mma1b = smem + mma1b_off(slot);
    uint8_t *kk = smem + kk_base(slot);
    const uint32_t kh = kk_half(slot);
    uint8_t *ga_c = smem + OFF_GA + (c0 >> 5) * GA_REGION;
    uint8_t *gb_c = smem + OFF_GB + (c0 >> 5) * GB_REGION;
    const uint32_t cb = (c0 & 31) * 4;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int r = 8 * qr + i;
        const float2 F = mul2(f[i], pre), G = mul2(gl[i], suf);
        // Gram operands, fp32 K-major (tf32 product): row = token (A: k rows 0..31, q rows
        // 32..63; B: k/F rows 0..31, tile-0 k*G rows 32..47), column = channel
        store_tf32x2(ga_c + sw128(r, cb), mul2(kv[i], F));                                  // K_L
        store_tf32x2(ga_c + sw128(32 + r, cb), mul2(qv[i], F));                             // Q_L
        store_tf32x2(gb_c + sw128(r, cb), mul2(kv[i], mul2(gl[i], ginv)));                // k/F
        if (tile == 0) store_tf32x2(gb_c + sw128(32 + r, cb), mul2(kv[i], G));              // k*G
    }
    // the Gram product can start (warp 2 issues it) while the operands of the state products
    // are written
    fence_proxy_async_smem();
    ok = gs.sync(misc) && ok;
    if (p == 0) mbar_arrive(&bars[B_GOPS_READY]);
    float qt0[8], qt1[8], kt0[8], kt1[8], kb0[8], kb1[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const float2 E = mul2(f[i], emul), X = mul2(gl[i], xmul);
        const float2 qt = mul2(qv[i], E), kt = mul2(kv[i], E), kb = mul2(kv[i], X);
        qt0[i] = qt.x; qt1[i] = qt.y; kt0[i] = kt.x; kt1[i] = kt.y; kb0[i] = kb.x; kb1[i] = kb.y;
    }
    // operands of the state products (one slot per step), 8 tokens = one 16-byte chunk per row
    store_chunk_f16(mma1b + sw128(c0, qr * 16), kt0);                // K~   (MMA1 B, N=r)
    store_chunk_f16(mma1b + sw128(c0 + 1, qr * 16), kt1);
    store_chunk_f16(mma1b + sw128(c0, (4 + qr) * 16), qt0);          // Q~   (MMA1 B, N=32+r)
    store_chunk_f16(mma1b + sw128(c0 + 1, (4 + qr) * 16), qt1);
    store_chunk_f16(kk + sw128(c0, kh + qr * 16), kb0);              // Kbar (R product A, k=r)
    store_chunk_f16(kk + sw128(c0 + 1, kh + qr * 16), kb1);
}

__device__ void prep_role(uint8_t *smem, uint64_t *bars, Misc *misc, int nsteps)
{
    const int p = threadIdx.x - 256;
    const long long start = misc->start, end = misc->end;
    GroupSync gs{2, 256};

    for (int s = 0; s < nsteps; ++s) {
        bool ok = true;
        const int qs = s % kQStages, slot = s % kSlots;
        const long long t0 = start + (long long)s * C;
        const int valid = (int)((end - t0) < C ? (end - t0) : C);
        if (s >= kSlots) wait_bar(&bars[B_OPS_FREE + slot], ((s / kSlots) - 1) & 1, misc);
        wait_bar(&bars[B_QFULL + qs], (s / kQStages) & 1, misc);
        if (p == 0) KDA_TRACE_EVENT(0, s);
        prep_operands(smem, smem + OFF_QRING + qs * QSTAGE_BYTES, p, slot, valid, misc, gs, ok,
                      bars, &bars[B_QEMPTY + qs], s);
        fence_proxy_async_smem();
        ok = gs.sync(misc) && ok;
        if (!ok) break;
        if (p == 0) {
            mbar_arrive(&bars[B_OPS_READY + slot]);   // MMA1 B, Kbar, b_C written
            KDA_TRACE_EVENT(2, s);
        }
    }
}

// ------------------------------------------------------------------------------------------------
// Two-warp block solve of T = (I + A)^-1 for the 32x32 strictly lower A, in 16x16 blocks:
//   T = [[T00, 0], [T10, T11]],  T00 = (I + A00)^-1,  T11 = (I + A11)^-1,  T10 = T11 (-A10) T00.
// Phase 1 (one warp): lane L < 16 forms column L of T00, lane L >= 16 column L-16 of T11, by a
// 16-row forward substitution.  Phase 2 (two warps, columns 0..7 and 8..15 of T10): M = (-A10) T00
// and T10 = T11 M, four rows per lane.  Shared memory holds -A (row stride 36) and, per step, T00
// by columns and T11 by rows.

constexpr uint32_t TB_BYTES = 2 * 16 * 16 * 4;   // T00 columns + T11 rows, fp32
static_assert(TB_BYTES == 2048, "shared-memory map reserves 2 KB per T-block buffer");

// column (lane & 15) of T00 (lanes 0..15) or of T11 (lanes 16..31)
__device__ __forceinline__ void solve_diag_blocks(const float *nA, int lane, float2 x2[8])
{
    const int base = (lane >> 4) * 16, c = lane & 15;
    if (!KDA_SMEM_OK(nA + base * 36 + base, (15 * 36 + 16) * 4, 12)) return;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const float *row = nA + (base + i) * 36 + base;
        float2 a01 = make_float2((i == c) ? 1.f : 0.f, 0.f), a23 = make_float2(0.f, 0.f);
#pragma unroll
        for (int m = 0; m < i / 4; ++m) {
            const float4 a4 = *reinterpret_cast<const float4 *>(row + 4 * m);
            a01 = fma2(make_float2(a4.x, a4.y), x2[2 * m], a01);
            a23 = fma2(make_float2(a4.z, a4.w), x2[2 * m + 1], a23);
        }
        if (i & 3) {
            const int q0 = 4 * (i / 4);
            const float4 a4 = *reinterpret_cast<const float4 *>(row + q0);
            a01.x = fmaf(a4.x, x2[q0 / 2].x, a01.x);
            if (i - q0 > 1) a01.y = fmaf(a4.y, x2[q0 / 2].y, a01.y);
            if (i - q0 > 2) a23.x = fmaf(a4.z, x2[q0 / 2 + 1].x, a23.x);
        }
        const float xi = (a01.x + a01.y) + (a23.x + a23.y);
        if (i & 1) x2[i / 2].y = xi; else x2[i / 2].x = xi;
    }
}

// rows 4*(lane>>3) .. +3 of column c = 8*half + (lane & 7) of T10
__device__ __forceinline__ void solve_offdiag(const float *nA, const float *tb, int half, int lane,
                                              float t10[4])
{
    const int c = 8 * half + (lane & 7), rq = lane >> 3;
    if (!KDA_SMEM_OK(tb, TB_BYTES, 13) || !KDA_SMEM_OK(nA + 16 * 36, 16 * 36 * 4, 14)) return;
    float2 tc[8];
#pragma unroll
    for (int g = 0; g < 4; ++g) {
        const float4 v = *reinterpret_cast<const float4 *>(tb + c * 16 + 4 * g);
        tc[2 * g] = make_float2(v.x, v.y);
        tc[2 * g + 1] = make_float2(v.z, v.w);
    }
    float m4[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const float *row = nA + (16 + 4 * rq + k) * 36;
        float2 a01 = make_float2(0.f, 0.f), a23 = make_float2(0.f, 0.f);
#pragma unroll
        for (int g = 0; g < 4; ++g) {
            const float4 a4 = *reinterpret_cast<const float4 *>(row + 4 * g);
            a01 = fma2(make_float2(a4.x, a4.y), tc[2 * g], a01);
            a23 = fma2(make_float2(a4.z, a4.w), tc[2 * g + 1], a23);
        }
        m4[k] = (a01.x + a01.y) + (a23.x + a23.y);
    }
    float2 mc[8];   // M[:, c] from the four lanes of column c
#pragma unroll
    for (int rr = 0; rr < 4; ++rr) {
        const int src = (lane & 7) + 8 * rr;
        mc[2 * rr] = make_float2(__shfl_sync(0xffffffffu, m4[0], src), __shfl_sync(0xffffffffu, m4[1], src));
        mc[2 * rr + 1] = make_float2(__shfl_sync(0xffffffffu, m4[2], src), __shfl_sync(0xffffffffu, m4[3], src));
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const float *row = tb + 256 + (4 * rq + k) * 16;
        float2 a01 = make_float2(0.f, 0.f), a23 = make_float2(0.f, 0.f);
#pragma unroll
        for (int g = 0; g < 4; ++g) {
            const float4 t4 = *reinterpret_cast<const float4 *>(row + 4 * g);
            a01 = fma2(make_float2(t4.x, t4.y), mc[2 * g], a01);
            a23 = fma2(make_float2(t4.z, t4.w), mc[2 * g + 1], a23);
        }
        t10[k] = (a01.x + a01.y) + (a23.x + a23.y);
    }
}

// phase 1 outputs: T00 columns and T11 rows to `tb`, and the Bt^T rows they fill
// (row c = beta_c T[:, c], fp16, bytes 64..127 of the AB slot's 128-byte rows)
__device__ __forceinline__ void store_diag_blocks(float *tb, uint8_t *ab, int lane, const float2 x2[8],
                                                  float bc)
{
    const int c = lane & 15;
    float t[8];
    if (!KDA_SMEM_OK(tb, TB_BYTES, 15)) return;
    if (lane < 16) {
#pragma unroll
        for (int g = 0; g < 4; ++g)
            *reinterpret_cast<float4 *>(tb + c * 16 + 4 * g) =
                make_float4(x2[2 * g].x, x2[2 * g].y, x2[2 * g + 1].x, x2[2 * g + 1].y);
#pragma unroll
        for (int m = 0; m < 2; ++m) {
#pragma unroll
            for (int i = 0; i < 4; ++i) { t[2 * i] = bc * x2[4 * m + i].x; t[2 * i + 1] = bc * x2[4 * m + i].y; }
            store_chunk_f16(ab + sw128(lane, 64 + 16 * m), t);    // rows 0..15 of column `lane`
        }
    } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            tb[256 + (2 * i) * 16 + c] = x2[i].x;
            tb[256 + (2 * i + 1) * 16 + c] = x2[i].y;
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) t[i] = 0.f;
        store_chunk_f16(ab + sw128(lane, 64), t);                 // rows 0..15: zero
        store_chunk_f16(ab + sw128(lane, 80), t);
#pragma unroll
        for (int m = 0; m < 2; ++m) {
#pragma unroll
            for (int i = 0; i < 4; ++i) { t[2 * i] = bc * x2[4 * m + i].x; t[2 * i + 1] = bc * x2[4 * m + i].y; }
            store_chunk_f16(ab + sw128(lane, 96 + 16 * m), t);    // rows 16..31 of column `lane`
        }
    }
}

// phase 2 output: rows 16 + 4*(lane>>3) .. +3 of Bt^T row c (fp16, one 8-byte store)
__device__ __forceinline__ void store_offdiag(uint8_t *ab, int half, int lane, const float t10[4], float bc)
{
    const int c = 8 * half + (lane & 7), rq = lane >> 3;
    const uint32_t lo = pack_f16x2(bc * t10[0], bc * t10[1]), hi = pack_f16x2(bc * t10[2], bc * t10[3]);
    if (KDA_SMEM_OK(ab + sw128(c, 96 + 8 * rq), 8, 16))
        *reinterpret_cast<uint2 *>(ab + sw128(c, 96 + 8 * rq)) = make_uint2(lo, hi);
}

// ------------------------------------------------------------------------------------------------
// Gram rows of a step: row r of the accumulator, column i of the 32 tokens.  Row tile 0 -> column
// i; row tile 1 -> column 32 + i for i in tile 0 (right operand relative to the end of tile 0),
// column i for i in tile 1.

struct GramRow {
    uint32_t r0[32], r1[16];
    __device__ __forceinline__ void load(uint32_t taddr)
    {
        tld32(taddr, r0);
        tld16(taddr + 32, r1);
        tmem_wait_ld();
    }
    __device__ __forceinline__ float at(int r, int i) const
    {
        return __uint_as_float((r >= 16 && i < 16) ? r1[i & 15] : r0[i & 31]);
    }
};

// warp 2: A = strict_lower(beta_r Gram_kk) (TMEM lanes 64..95) into shared memory (negated) for the
// solver warps, with beta, which this warp loads one step ahead.

__device__ void a_role(const Params &p, uint8_t *smem, uint64_t *bars, Misc *misc, int h, int nsteps)
{
    const int lane = threadIdx.x & 31;
    const uint32_t tb = misc->tmem_base + ((uint32_t)64 << 16);
    float *sA = reinterpret_cast<float *>(smem + OFF_SA);
    float *sbeta_all = reinterpret_cast<float *>(smem + OFF_BETA);
    const long long start = misc->start, end = misc->end;
    auto load_beta = [&](int t) -> float {
        const long long tok = start + (long long)t * C + lane;
        return tok < end ? __bfloat162float(p.beta[tok * p.H + h]) : 0.f;
    };
    float bnext = load_beta(0);
    for (int s = 0; s < nsteps; ++s) {
        const int buf = s & 1;
        // the Gram of the step: its operands are written, and the accumulator of this parity was
        // read two steps ago
        if (lane == 0) {
            bool go = wait_bar(&bars[B_GOPS_READY], s & 1, misc);
            if (go && s >= 2) go = wait_bar(&bars[B_EXTR_DONE + buf], ((s >> 1) - 1) & 1, misc);
            if (go) {
                tc_fence_after();
                issue_gram(misc->tmem_base, smem_u32(smem), buf, &bars[B_GRAM_DONE + buf]);
            }
        }
        __syncwarp();
        const float br = bnext;
        if (s + 1 < nsteps) bnext = load_beta(s + 1);
        bool ok = wait_bar(&bars[B_GRAM_DONE + buf], (s >> 1) & 1, misc);
        if (s >= 1) ok = wait_bar(&bars[B_SA_FREE], (s - 1) & 1, misc) && ok;   // A of s-1 read
        if (!__all_sync(0xffffffffu, ok)) break;
        if (lane == 0) KDA_TRACE_EVENT(4, s);
        tc_fence_after();
        GramRow g;
        g.load(tb + TM_DG + 48 * buf);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[B_EXTR_DONE + buf]);
        const int r = lane;   // token row
        // (a failed debug check skips the stores; the warp stays on its path)
        const bool st_ok = KDA_SMEM_OK(sA + r * 36, 128, 10) && KDA_SMEM_OK(sbeta_all + buf * C + r, 4, 11);
        if (st_ok) sbeta_all[buf * C + r] = br;
        const float nbr = -br;           // sA holds -A
#pragma unroll
        for (int m = 0; m < 8; ++m) {
            float4 v;
            v.x = (4 * m + 0 < r) ? nbr * g.at(r, 4 * m + 0) : 0.f;
            v.y = (4 * m + 1 < r) ? nbr * g.at(r, 4 * m + 1) : 0.f;
            v.z = (4 * m + 2 < r) ? nbr * g.at(r, 4 * m + 2) : 0.f;
            v.w = (4 * m + 3 < r) ? nbr * g.at(r, 4 * m + 3) : 0.f;
            if (st_ok) *reinterpret_cast<float4 *>(sA + r * 36 + 4 * m) = v;
        }
        __syncwarp();
        if (lane == 0) {
            mbar_arrive(&bars[B_A_READY]);
            KDA_TRACE_EVENT(5, s);
        }
    }
    if (lane == 0) drain_mmas(&bars[B_DRAIN + 1], misc);
}

// solver warps.  Warp 1: phase 1 of the block solve (T00, T11) and half 0 of phase 2; warp 3: Aqk
// = lower_incl_diag(Gram_qk) (TMEM lanes 96..127) into the P product's A operand, and half 1 of
// phase 2.  Together they write Bt^T = (T diag(beta))^T (fp16, the B operand of the P and R
// products, which the issuer starts once both have signalled).

__device__ void solver_role(uint8_t *smem, uint64_t *bars, Misc *misc, int nsteps, int half)
{
    const int lane = threadIdx.x & 31;
    const float *nA = reinterpret_cast<const float *>(smem + OFF_SA);
    const float *sbeta_all = reinterpret_cast<const float *>(smem + OFF_BETA);
    for (int s = 0; s < nsteps; ++s) {
        const int buf = s & 1, slot = s % kSlots;
        float *tblk = reinterpret_cast<float *>(smem + OFF_TB + buf * TB_BYTES);
        uint8_t *ab = smem + ab_off(slot);
        bool ok;
        if (half == 0) {
            ok = wait_bar(&bars[B_A_READY], s & 1, misc);
            if (!__all_sync(0xffffffffu, ok)) break;
            if (lane == 0) KDA_TRACE_EVENT(6, s);
            float2 x2[8];
            solve_diag_blocks(nA, lane, x2);
            store_diag_blocks(tblk, ab, lane, x2, -sbeta_all[buf * C + lane]);
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&bars[B_T_READY + buf]);   // T00 and T11 for the other half of phase 2
                KDA_TRACE_EVENT(7, s);
            }
        } else {
            // Aqk of the step (q-rows of the Gram)
            ok = wait_bar(&bars[B_GRAM_DONE + buf], (s >> 1) & 1, misc);
            if (!__all_sync(0xffffffffu, ok)) break;
            tc_fence_after();
            GramRow g;
            g.load(misc->tmem_base + ((uint32_t)96 << 16) + TM_DG + 48 * buf);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[B_EXTR_DONE + buf]);
            const int r = lane;
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                float t[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) t[i] = (8 * m + i <= r) ? g.at(r, 8 * m + i) : 0.f;
                store_chunk_f16(ab + sw128(r, m * 16), t);          // Aqk row r
#if KDA_PRECISE
#pragma unroll
                for (int i = 0; i < 8; ++i) t[i] -= __half2float(__float2half_rn(t[i]));   // exact in fp32
                store_chunk_f16(smem + alo_rows(slot) + sw128(r, alo_half(slot) + m * 16), t);   // Aqk_lo
#endif
            }
            ok = wait_bar(&bars[B_T_READY + buf], (s >> 1) & 1, misc);
            if (!__all_sync(0xffffffffu, ok)) break;
        }
        float t10[4];
        solve_offdiag(nA, tblk, half, lane, t10);
        const float bc = -sbeta_all[buf * C + 8 * half + (lane & 7)];
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[B_SA_FREE]);   // A and beta of the step read
        store_offdiag(ab, half, lane, t10, bc);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
            mbar_arrive(&bars[B_BT_READY + slot]);     // this warp's part of Aqk and Bt written
            if (half == 0) KDA_TRACE_EVENT(8, s);
        }
        if (__any_sync(0xffffffffu, misc->abort != 0)) break;
    }
}

// ------------------------------------------------------------------------------------------------
// asynchronous issuer (lane 0 of warp 0): every TMA load, and the chain's V products, state reads
// and P / R^T products, each issued as soon as its inputs are ready.  The q, k, g load goes first
// in every round: its single stage is the loop prep waits on (prep -> release -> load -> prep),
// so it is released per warp as soon as the values are in registers and reissued at once.  The
// barriers are polled without blocking, so that no ready operation waits behind another one;
// every condition below is checked only after its previous phase has been observed, so a parity
// test is never ahead.

__device__ void issuer_role(const Params &p, const CUtensorMap *mq, const CUtensorMap *mk,
                            const CUtensorMap *mg, const CUtensorMap *mv, uint8_t *smem,
                            uint64_t *bars, Misc *misc, int h, int nsteps)
{
    const uint32_t tm = misc->tmem_base;
    const uint32_t sb = smem_u32(smem);
    const long long start = misc->start;
    const CUtensorMap *maps[3] = {mq, mk, mg};
    int sq = 0, sv = 0, cvi = 0, c1 = 0, cp = 0;
    long long last = clock64();
    while (c1 < nsteps || cp < nsteps) {
        bool prog = false;
        // q, k, g of step sq (one stage: free once prep holds step sq-1 in registers)
        if (sq < nsteps && (sq == 0 || mbar_test_wait(&bars[B_QEMPTY], (sq - 1) & 1))) {
            const int t0 = (int)(start + (long long)sq * C);
            mbar_arrive_expect_tx(&bars[B_QFULL], QSTAGE_BYTES);
#pragma unroll
            for (int x = 0; x < 3; ++x)
#pragma unroll
                for (int half = 0; half < 2; ++half)
                    tma_load_3d(smem + OFF_QRING + x * TILE_BYTES + half * 4096, maps[x], &bars[B_QFULL],
                                half * 64, h, t0);
            KDA_TRACE_EVENT(19, sq);
            ++sq;
            prog = true;
        }
        // the chain's products first (they are on its critical path), then the loads
        // state reads of step c1: after its V product, the chain's fp16 state copy and prep's
        // operands
        if (c1 < cvi && mbar_test_wait(&bars[B_SBF_READY], c1 & 1) &&
            mbar_test_wait(&bars[B_OPS_READY + c1 % kSlots], (c1 / kSlots) & 1)) {
            KDA_TRACE_EVENT(21, c1);
            tc_fence_after();
            issue_mma1(tm, sb, c1 & 1, c1 % kSlots, &bars[B_MMA1_DONE]);
            KDA_TRACE_EVENT(20, c1);
            ++c1;
            prog = true;
        }
        // P and R^T of step cp: Bt from the solver, and the chain read those of step cp-1
        if (cp < nsteps && mbar_test_wait(&bars[B_BT_READY + cp % kSlots], (cp / kSlots) & 1) &&
            (cp == 0 || mbar_test_wait(&bars[B_PR_FREE], (cp - 1) & 1))) {
            tc_fence_after();
            issue_pr(tm, sb, cp % kSlots, &bars[B_PR_DONE]);
            KDA_TRACE_EVENT(3, cp);
            ++cp;
            prog = true;
        }
        // V product of step cvi: its v landed, and the chain read the outputs of step cvi-2
        if (cvi < sv && mbar_test_wait(&bars[B_VFULL + cvi % kVStages], (cvi / kVStages) & 1) &&
            (cvi < 2 || mbar_test_wait(&bars[B_D1_FREE + (cvi & 1)], ((cvi - 2) >> 1) & 1))) {
            tc_fence_after();
            issue_vi(tm, sb, cvi & 1, cvi % kVStages);
            KDA_TRACE_EVENT(22, cvi);
            ++cvi;
            prog = true;
        }
        // v of step sv (kVStages stages: free once the V product of step sv - kVStages has completed)
        if (sv < nsteps && (sv < kVStages || mbar_test_wait(&bars[B_VEMPTY + sv % kVStages], ((sv / kVStages) - 1) & 1))) {
            const int t0 = (int)(start + (long long)sv * C);
            uint8_t *vt = smem + OFF_VRING + (sv % kVStages) * TILE_BYTES;
            mbar_arrive_expect_tx(&bars[B_VFULL + sv % kVStages], TILE_BYTES);
#pragma unroll
            for (int half = 0; half < 2; ++half)
                tma_load_3d(vt + half * 4096, mv, &bars[B_VFULL + sv % kVStages], half * 64, h, t0);
            KDA_TRACE_EVENT(18, sv);
            ++sv;
            prog = true;
        }
        if (prog) {
            last = clock64();
        } else {
            if (misc->abort) break;
            if (clock64() - last > kTimeout) {
                fail(misc);
                break;
            }
            __nanosleep(32);
        }
    }
    // never leave the CTA with copies or products in flight
    if (sq > 0) mbar_wait(&bars[B_QFULL], (sq - 1) & 1, &misc->zero, kTimeout);
    for (int t = (sv > kVStages ? sv - kVStages : 0); t < sv; ++t)
        mbar_wait(&bars[B_VFULL + t % kVStages], (t / kVStages) & 1, &misc->zero, kTimeout);
    drain_mmas(&bars[B_DRAIN + 2], misc);
}

template <typename TO>
__global__ void __launch_bounds__(kThreads, 1)
prefill_tc_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
                  const __grid_constant__ CUtensorMap mg, const __grid_constant__ CUtensorMap mv,
                  const __grid_constant__ CUtensorMap mo, const Params p)
{
    extern __shared__ __align__(16) uint8_t smem_raw[];
    // 1024-byte aligned base by pointer arithmetic on the shared array, so that the compiler keeps
    // every access through `smem` in the shared state space (an integer round trip would turn
    // them into generic loads and stores)
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + OFF_BARS);
    Misc *misc = reinterpret_cast<Misc *>(smem + OFF_MISC);
    const int warp = threadIdx.x >> 5;
    const int h = blockIdx.x % p.H;

    select_item(p, misc);
    if (threadIdx.x == 0) {
        for (int s = 0; s < kQStages; ++s) {
            mbar_init(&bars[B_QFULL + s], 1);        // the expect_tx arrival
            mbar_init(&bars[B_QEMPTY + s], 8);        // one arrival per prep warp
        }
        for (int s = 0; s < kVStages; ++s) {
            mbar_init(&bars[B_VFULL + s], 1);        // the expect_tx arrival
            mbar_init(&bars[B_VEMPTY + s], 1);
        }
        for (int b = B_OPS_READY; b < B_COUNT; ++b) mbar_init(&bars[b], 1);
        for (int b = 0; b < 2; ++b) mbar_init(&bars[B_EXTR_DONE + b], 2);   // warps 2 and 3
        mbar_init(&bars[B_SA_FREE], 2);                                      // solver warps 1 and 3
        for (int b = 0; b < kSlots; ++b) mbar_init(&bars[B_BT_READY + b], 2);
        static_assert(B_VEMPTY >= B_VFULL + kVStages && B_OPS_READY >= B_VEMPTY + kVStages, "barrier layout");
        fence_barrier_init();
    }
    if (warp == 0) {
        tma_prefetch_desc(&mq); tma_prefetch_desc(&mk); tma_prefetch_desc(&mg); tma_prefetch_desc(&mv);
    }
    if (warp == 1) {
        tmem_alloc(&misc->tmem_base, TM_COLS);
        tmem_relinquish();
    }
    // the constant B operand [-I | 0] of the V product (bf16, rows n = 0..63, K = 32 tokens)
    for (int e = threadIdx.x; e < 64 * 16; e += kThreads) {
        const int row = e >> 4, wd = e & 15;
        const uint32_t lo = (row == 2 * wd) ? 0xBF80u : 0u, hi = (row == 2 * wd + 1) ? 0xBF80u : 0u;
        *reinterpret_cast<uint32_t *>(smem + kk_base(kEyeSlot) + sw128(row, kk_half(kEyeSlot) + 4 * wd)) =
            lo | (hi << 16);
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
        if (threadIdx.x == 0) issuer_role(p, &mq, &mk, &mg, &mv, smem, bars, misc, h, nsteps);
    } else if (warp == 1 || warp == 3) {
        solver_role(smem, bars, misc, nsteps, warp == 3);
    } else if (warp == 2) {
        a_role(p, smem, bars, misc, h, nsteps);
    } else if (warp < 8) {
        chain_role<TO>(p, &mo, smem, bars, misc, h, nsteps);
    } else {
        prep_role(smem, bars, misc, nsteps);
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

// output tiles: [T, H, 128] of fp32 or bf16, box = 128 channels x 1 head x 32 tokens, unswizzled
bool make_out_map(CUtensorMap *map, void *base, int H, int64_t T, bool f32)
{
    auto enc = encode_fn();
    if (!enc) return false;
    const cuuint64_t es = f32 ? 4 : 2;
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)T};
    cuuint64_t strides[2] = {(cuuint64_t)D * es, (cuuint64_t)H * D * es};
    cuuint32_t box[3] = {(cuuint32_t)D, 1, (cuuint32_t)C}, estr[3] = {1, 1, 1};
    return enc(map, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base, dims,
               strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
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
                 const CUtensorMap &mv, const CUtensorMap &mo, const Params &p, int blocks,
                 cudaStream_t stream)
{
    // a function attribute belongs to the current device: set it on every launch
    if (cudaFuncSetAttribute(prefill_tc_kernel<TO>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             SMEM_ALLOC) != cudaSuccess)
        return KDA_ERR_CUDA;
    prefill_tc_kernel<TO><<<blocks, kThreads, SMEM_ALLOC, stream>>>(mq, mk, mg, mv, mo, p);
    return cudaGetLastError() == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

}  // namespace

#if !KDA_PRECISE
namespace {

// One CTA whose bounded wait is on a barrier that nothing ever completes: the same wait the prefill
// kernel uses gives up after `cycles` SM cycles and records the timeout in the device error word.
__global__ void wait_timeout_probe_kernel(long long cycles)
{
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0 && !mbar_wait(&bar, 0, &abort_flag, cycles))
        atomicExch(&g_prefill_tc_error, KDA_ERR_DEVICE_TIMEOUT);
}

}  // namespace

// One thread runs the shared-memory bounds check on an offset past its CTA's window (nothing is
// accessed): the check records KDA_ERR_DEVICE_BOUNDS, as a failed check in a debug build would.
__global__ void bounds_check_probe_kernel()
{
    (void)smem_in_window(kda_dyn_smem + SMEM_ALLOC, 16, 99);
}

int launch_bounds_check_probe(cudaStream_t stream)
{
    bounds_check_probe_kernel<<<1, 1, 0, stream>>>();
    return cudaGetLastError() == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

int launch_wait_timeout_probe(long long cycles, cudaStream_t stream)
{
    wait_timeout_probe_kernel<<<1, 32, 0, stream>>>(cycles);
    return cudaGetLastError() == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}
#endif

int KDA_TC_EXPORT(read_and_clear_debug_site)(cudaStream_t s, int32_t *site)
{
    int host = 0, zero = 0;
    if (cudaMemcpyFromSymbolAsync(&host, g_prefill_tc_debug_site, sizeof(int), 0, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaMemcpyToSymbolAsync(g_prefill_tc_debug_site, &zero, sizeof(int), 0, cudaMemcpyHostToDevice, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return KDA_ERR_CUDA;
    *site = host;
    return KDA_OK;
}

int KDA_TC_EXPORT(read_and_clear_status_prefill_tc)(cudaStream_t s, int32_t *status)
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

int KDA_TC_EXPORT(launch_prefill_tc)(const void *q, const void *k, const void *v, const void *g,
                      const void *beta, const int32_t *cu_seqlens, int n_seqs,
                      int64_t total_tokens, int n_heads, int out_dtype, const float *init_state,
                      void *out, float *final_state, int ckpt_stride, float *ckpts,
                      cudaStream_t stream)
{
    const int64_t blocks = (int64_t)n_seqs * n_heads;
    if (blocks == 0) return KDA_OK;
    if (blocks > 0x7fffffffLL) return KDA_ERR_INVALID_ARG;
    CUtensorMap mq, mk, mg, mv, mo;
    if (!make_map(&mq, q, n_heads, total_tokens) || !make_map(&mk, k, n_heads, total_tokens) ||
        !make_map(&mg, g, n_heads, total_tokens) || !make_map(&mv, v, n_heads, total_tokens) ||
        !make_out_map(&mo, out, n_heads, total_tokens, out_dtype != KDA_BF16))
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
    if (out_dtype == KDA_BF16) return launch_typed<__nv_bfloat16>(mq, mk, mg, mv, mo, p, (int)blocks, stream);
    return launch_typed<float>(mq, mk, mg, mv, mo, p, (int)blocks, stream);
}

#if defined(KDA_TRACE) && !KDA_PRECISE
extern "C" int kda_trace_read(long long *dst)
{
    return cudaMemcpyFromSymbol(dst, g_kda_trace, sizeof(g_kda_trace)) == cudaSuccess ? 0 : 1;
}
#endif

}  // namespace kda
