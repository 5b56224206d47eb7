// kda_capi.cu -- the C ABI of libkda_gb300: host-side argument validation and kernel dispatch.
// Declarations, argument meaning, layouts and error behaviour: include/kda.h.
#include <cstdio>

#include <nvtx3/nvToolsExt.h>

#include "kda_internal.cuh"

using namespace kda;

namespace {

// An NVTX range over one C-ABI call, so that profiler captures can be scoped to a call.  Without
// a tool attached the push and pop do nothing.
struct CallRange {
    explicit CallRange(const char *name) { nvtxRangePushA(name); }
    ~CallRange() { nvtxRangePop(); }
    CallRange(const CallRange &) = delete;
    CallRange &operator=(const CallRange &) = delete;
};

bool bad_dtype(int32_t dtype) { return dtype != KDA_BF16 && dtype != KDA_F32; }

// Validation shared by both prefill entry points.  Returns KDA_OK when the call may launch.
int check_prefill(const void *q, const void *k, const void *v, const void *g, const void *beta,
                  const int32_t *cu_seqlens, int32_t n_seqs, int64_t total_tokens, int32_t n_heads,
                  int32_t d_k, int32_t d_v, int32_t dtype, int32_t out_dtype,
                  const float *init_state, const void *out, const float *final_state,
                  int32_t ckpt_stride, const float *ckpts)
{
    if (n_seqs < 0 || total_tokens < 0 || n_heads < 1 || d_k < 1 || d_v < 1 || bad_dtype(dtype) ||
        bad_dtype(out_dtype))
        return KDA_ERR_INVALID_ARG;
    if (total_tokens > 0 && (!q || !k || !v || !g || !beta || !out)) return KDA_ERR_INVALID_ARG;
    if (total_tokens > 0 && n_seqs == 0) return KDA_ERR_INVALID_ARG;
    if (!cu_seqlens && n_seqs > 1) return KDA_ERR_INVALID_ARG;
    if (total_tokens > 0x7fffffffLL) return KDA_ERR_INVALID_ARG;  // cu_seqlens are int32
    // a checkpoint falls on a boundary of the tensor-core kernel's 32-token steps
    if (ckpt_stride < 0 || ckpt_stride % 32 != 0) return KDA_ERR_INVALID_ARG;
    if (ckpt_stride > 0 && !ckpts) return KDA_ERR_INVALID_ARG;
    const void *ptrs[] = {q, k, v, g, beta, init_state, out, final_state, ckpts};
    for (const void *p : ptrs)
        if (p && !aligned16(p)) return KDA_ERR_MISALIGNED;
    if ((reinterpret_cast<uintptr_t>(cu_seqlens) & 3u) != 0) return KDA_ERR_MISALIGNED;
    const int esz = dtype == KDA_BF16 ? 2 : 4, osz = out_dtype == KDA_BF16 ? 2 : 4;
    // every row of q/k/g/v/out must start 16-byte aligned for the vector and TMA paths
    if (((int64_t)d_k * esz) % 16 != 0 || ((int64_t)d_v * esz) % 16 != 0 ||
        ((int64_t)d_v * osz) % 16 != 0)
        return KDA_ERR_UNSUPPORTED_SHAPE;
    if (out && (out == q || out == k || out == v || out == g || out == beta))
        return KDA_ERR_INVALID_ARG;
    return KDA_OK;
}

// Validation shared by the two staged entry points (everything but the scratch).
int check_staged(const void *h_q, const void *h_k, const void *h_v, const void *h_g, const void *h_beta,
                 const int32_t *h_cu_seqlens, int32_t n_seqs, int64_t total_tokens, int32_t n_heads,
                 int32_t dtype, int32_t out_dtype, const float *init_state, void *d_q, void *d_k,
                 void *d_v, void *d_g, void *d_beta, void *d_out, void *h_out, float *final_state,
                 int64_t chunk_tokens)
{
    if (n_seqs < 0 || total_tokens < 0 || n_heads < 1 || chunk_tokens < 1 || bad_dtype(dtype) ||
        bad_dtype(out_dtype) || total_tokens > 0x7fffffffLL)
        return KDA_ERR_INVALID_ARG;
    if ((total_tokens > 0 && n_seqs == 0) || (n_seqs > 0 && !final_state) || (n_seqs > 1 && !h_cu_seqlens))
        return KDA_ERR_INVALID_ARG;
    const void *host_in[] = {h_q, h_k, h_v, h_g, h_beta, h_out};
    const void *dev_buf[] = {d_q, d_k, d_v, d_g, d_beta, d_out};
    for (int i = 0; i < 6; ++i)
        if (total_tokens > 0 && (!host_in[i] || !dev_buf[i])) return KDA_ERR_INVALID_ARG;
    const void *ptrs[] = {h_q, h_k, h_v, h_g, h_beta, h_out, d_q, d_k, d_v, d_g, d_beta, d_out,
                          init_state, final_state};
    for (const void *p : ptrs)
        if (p && !aligned16(p)) return KDA_ERR_MISALIGNED;
    // every chunk after the first starts at a multiple of chunk_tokens (or of 32 in the cut-up
    // last chunk), and its beta rows must start 16-byte aligned like every pointer of a prefill
    const int64_t esz = dtype == KDA_BF16 ? 2 : 4;
    if (total_tokens > chunk_tokens && (chunk_tokens * n_heads * esz) % 16 != 0) return KDA_ERR_INVALID_ARG;
    if (n_seqs > 1) {   // the host table is checked in full here
        if (h_cu_seqlens[0] != 0 || h_cu_seqlens[n_seqs] != total_tokens) return KDA_ERR_INVALID_ARG;
        for (int n = 0; n < n_seqs; ++n)
            if (h_cu_seqlens[n + 1] < h_cu_seqlens[n]) return KDA_ERR_INVALID_ARG;
    }
    return KDA_OK;
}

bool tc_supported(int32_t d_k, int32_t d_v, int32_t dtype)
{
    return dtype == KDA_BF16 && d_k == 128 && d_v == 128;
}

}  // namespace

extern "C" {

int kda_abi_version(void) { return KDA_ABI_VERSION; }

const char *kda_status_string(int status)
{
    switch (status) {
    case KDA_OK: return "KDA_OK";
    case KDA_ERR_INVALID_ARG: return "KDA_ERR_INVALID_ARG: invalid argument";
    case KDA_ERR_UNSUPPORTED_SHAPE: return "KDA_ERR_UNSUPPORTED_SHAPE: head sizes not implemented";
    case KDA_ERR_MISALIGNED: return "KDA_ERR_MISALIGNED: pointer not 16-byte aligned";
    case KDA_ERR_CUDA: return "KDA_ERR_CUDA: CUDA runtime call or launch failed";
    case KDA_ERR_DEVICE_TIMEOUT: return "KDA_ERR_DEVICE_TIMEOUT: bounded device wait expired";
    case KDA_ERR_INDEX_RANGE: return "KDA_ERR_INDEX_RANGE: state index out of range";
    case KDA_ERR_DEVICE_BOUNDS: return "KDA_ERR_DEVICE_BOUNDS: device-side bounds check failed";
    default: return "KDA_ERR_UNKNOWN";
    }
}

int kda_prefill_path(int32_t d_k, int32_t d_v, int32_t dtype)
{
    if (d_k < 1 || d_v < 1 || bad_dtype(dtype)) return -KDA_ERR_INVALID_ARG;
    if (tc_supported(d_k, d_v, dtype)) return 1;
    if (d_k <= 128 && d_v % 32 == 0 && d_v <= 256) return 0;
    return -KDA_ERR_UNSUPPORTED_SHAPE;
}

int kda_prefill(const void *q, const void *k, const void *v, const void *g, const void *beta,
                const int32_t *cu_seqlens, int32_t n_seqs, int64_t total_tokens, int32_t n_heads,
                int32_t d_k, int32_t d_v, int32_t dtype, int32_t out_dtype, const float *init_state,
                void *out, float *final_state, int32_t ckpt_stride, float *ckpts, void *stream)
{
    const CallRange range("kda_prefill");
    int rc = check_prefill(q, k, v, g, beta, cu_seqlens, n_seqs, total_tokens, n_heads, d_k, d_v,
                           dtype, out_dtype, init_state, out, final_state, ckpt_stride, ckpts);
    if (rc != KDA_OK) return rc;
    if (tc_supported(d_k, d_v, dtype) && total_tokens > 0)
        return launch_prefill_tc(q, k, v, g, beta, cu_seqlens, n_seqs, total_tokens, n_heads,
                                 out_dtype, init_state, out, final_state, ckpt_stride, ckpts,
                                 (cudaStream_t)stream);
    return launch_prefill_recurrent(q, k, v, g, beta, cu_seqlens, n_seqs, total_tokens, n_heads,
                                    d_k, d_v, dtype, out_dtype, init_state, out, final_state,
                                    ckpt_stride, ckpts, (cudaStream_t)stream);
}

int kda_prefill_precise(const void *q, const void *k, const void *v, const void *g,
                        const void *beta, const int32_t *cu_seqlens, int32_t n_seqs,
                        int64_t total_tokens, int32_t n_heads, int32_t d_k, int32_t d_v,
                        int32_t dtype, int32_t out_dtype, const float *init_state, void *out,
                        float *final_state, int32_t ckpt_stride, float *ckpts, void *stream)
{
    const CallRange range("kda_prefill_precise");
    int rc = check_prefill(q, k, v, g, beta, cu_seqlens, n_seqs, total_tokens, n_heads, d_k, d_v,
                           dtype, out_dtype, init_state, out, final_state, ckpt_stride, ckpts);
    if (rc != KDA_OK) return rc;
    if (tc_supported(d_k, d_v, dtype) && total_tokens > 0)
        return launch_prefill_tc_precise(q, k, v, g, beta, cu_seqlens, n_seqs, total_tokens,
                                         n_heads, out_dtype, init_state, out, final_state,
                                         ckpt_stride, ckpts, (cudaStream_t)stream);
    return launch_prefill_recurrent(q, k, v, g, beta, cu_seqlens, n_seqs, total_tokens, n_heads,
                                    d_k, d_v, dtype, out_dtype, init_state, out, final_state,
                                    ckpt_stride, ckpts, (cudaStream_t)stream);
}

int kda_prefill_recurrent(const void *q, const void *k, const void *v, const void *g,
                          const void *beta, const int32_t *cu_seqlens, int32_t n_seqs,
                          int64_t total_tokens, int32_t n_heads, int32_t d_k, int32_t d_v,
                          int32_t dtype, int32_t out_dtype, const float *init_state, void *out,
                          float *final_state, int32_t ckpt_stride, float *ckpts, void *stream)
{
    const CallRange range("kda_prefill_recurrent");
    int rc = check_prefill(q, k, v, g, beta, cu_seqlens, n_seqs, total_tokens, n_heads, d_k, d_v,
                           dtype, out_dtype, init_state, out, final_state, ckpt_stride, ckpts);
    if (rc != KDA_OK) return rc;
    return launch_prefill_recurrent(q, k, v, g, beta, cu_seqlens, n_seqs, total_tokens, n_heads,
                                    d_k, d_v, dtype, out_dtype, init_state, out, final_state,
                                    ckpt_stride, ckpts, (cudaStream_t)stream);
}

int kda_decode(const void *q, const void *k, const void *v, const void *g, const void *beta,
               float *state, void *out, int32_t n_seqs, int32_t n_heads, int32_t d_k, int32_t d_v,
               int32_t dtype, int32_t out_dtype, void *stream)
{
    const CallRange range("kda_decode");
    if (n_seqs < 0 || n_heads < 1 || d_k < 1 || d_v < 1 || bad_dtype(dtype) || bad_dtype(out_dtype))
        return KDA_ERR_INVALID_ARG;
    if (n_seqs > 0 && (!q || !k || !v || !g || !beta || !state || !out)) return KDA_ERR_INVALID_ARG;
    const void *ptrs[] = {q, k, v, g, beta, state, out};
    for (const void *p : ptrs)
        if (p && !aligned16(p)) return KDA_ERR_MISALIGNED;
    if (out && (out == q || out == k || out == v || out == g || out == beta || out == state))
        return KDA_ERR_INVALID_ARG;
    return launch_decode(q, k, v, g, beta, state, out, n_seqs, n_heads, d_k, d_v, dtype, out_dtype,
                         (cudaStream_t)stream);
}

int kda_state_copy(float *dst, const int64_t *dst_idx, int64_t n_dst_slots, const float *src,
                   const int64_t *src_idx, int64_t n_src_slots, int64_t n, int32_t n_heads,
                   int32_t d_k, int32_t d_v, void *stream)
{
    const CallRange range("kda_state_copy");
    if (n < 0 || n_dst_slots < 0 || n_src_slots < 0 || n_heads < 1 || d_k < 1 || d_v < 1)
        return KDA_ERR_INVALID_ARG;
    if (n > 0 && (!dst || !src)) return KDA_ERR_INVALID_ARG;
    if ((!dst_idx && n > n_dst_slots) || (!src_idx && n > n_src_slots)) return KDA_ERR_INVALID_ARG;
    const void *ptrs[] = {dst, dst_idx, src, src_idx};
    for (const void *p : ptrs)
        if (p && !aligned16(p)) return KDA_ERR_MISALIGNED;
    const int64_t unit = (int64_t)n_heads * d_k * d_v;
    return launch_state_copy(dst, dst_idx, n_dst_slots, src, src_idx, n_src_slots, n, unit,
                             (cudaStream_t)stream);
}

int kda_premix(const void *xq, const void *xk, const void *xv, const void *a, const void *b,
               const float *w, const void *hist, const int32_t *cu_seqlens, int32_t n_seqs,
               int64_t total_tokens, int32_t n_heads, int32_t d, float eps, int32_t dtype, void *q,
               void *k, void *v, void *g, void *beta, void *stream)
{
    const CallRange range("kda_premix");
    if (n_seqs < 0 || total_tokens < 0 || n_heads < 1 || d < 1 || bad_dtype(dtype) || !(eps > 0.f))
        return KDA_ERR_INVALID_ARG;
    if (total_tokens > 0 && n_seqs == 0) return KDA_ERR_INVALID_ARG;
    if (total_tokens > 0x7fffffffLL) return KDA_ERR_INVALID_ARG;   // cu_seqlens are int32
    if (!cu_seqlens && n_seqs > 1) return KDA_ERR_INVALID_ARG;
    if (total_tokens > 0 && (!xq || !xk || !xv || !a || !b || !w || !q || !k || !v || !g || !beta))
        return KDA_ERR_INVALID_ARG;
    if (d > 256 || (d & (d - 1)) != 0 || d < 8) return KDA_ERR_UNSUPPORTED_SHAPE;
    const void *ptrs[] = {xq, xk, xv, a, b, w, hist, q, k, v, g, beta};
    for (const void *p : ptrs)
        if (p && !aligned16(p)) return KDA_ERR_MISALIGNED;
    if ((reinterpret_cast<uintptr_t>(cu_seqlens) & 3u) != 0) return KDA_ERR_MISALIGNED;
    const void *ins[] = {xq, xk, xv, a, b, hist};
    const void *outs[] = {q, k, v, g, beta};
    for (const void *o : outs)
        for (const void *i : ins)
            if (o && o == i) return KDA_ERR_INVALID_ARG;
    return launch_premix(xq, xk, xv, a, b, w, hist, cu_seqlens, n_seqs, total_tokens, n_heads, d,
                         eps, dtype, q, k, v, g, beta, (cudaStream_t)stream);
}

int kda_output_gate(const void *o, int32_t o_dtype, const void *z, int32_t z_dtype, void *out,
                    int32_t out_dtype, int64_t n, void *stream)
{
    const CallRange range("kda_output_gate");
    if (n < 0 || bad_dtype(o_dtype) || bad_dtype(z_dtype) || bad_dtype(out_dtype))
        return KDA_ERR_INVALID_ARG;
    if (n > 0 && (!o || !z || !out)) return KDA_ERR_INVALID_ARG;
    const void *ptrs[] = {o, z, out};
    for (const void *p : ptrs)
        if (p && !aligned16(p)) return KDA_ERR_MISALIGNED;
    // in place over o is fine (same element type: each element is read before it is written)
    if (out && ((out == o && out_dtype != o_dtype) || out == z)) return KDA_ERR_INVALID_ARG;
    return launch_output_gate(o, o_dtype, z, z_dtype, out, out_dtype, n, (cudaStream_t)stream);
}

int kda_cp_combine(const float *s_loc, const float *m, const int32_t *seq_seg, int32_t n_seqs,
                   int32_t n_heads, int32_t d, float *s_start, float *final_state, void *stream)
{
    const CallRange range("kda_cp_combine");
    if (n_seqs < 0 || n_heads < 1 || d < 1) return KDA_ERR_INVALID_ARG;
    if (d != 128) return KDA_ERR_UNSUPPORTED_SHAPE;
    if (n_seqs > 0 && (!s_loc || !m || !seq_seg || !s_start)) return KDA_ERR_INVALID_ARG;
    const void *ptrs[] = {s_loc, m, s_start, final_state};
    for (const void *p : ptrs)
        if (p && !aligned16(p)) return KDA_ERR_MISALIGNED;
    if ((reinterpret_cast<uintptr_t>(seq_seg) & 3u) != 0) return KDA_ERR_MISALIGNED;
    if (s_start && (s_start == s_loc || s_start == m)) return KDA_ERR_INVALID_ARG;
    if (final_state && (final_state == s_loc || final_state == m || final_state == s_start))
        return KDA_ERR_INVALID_ARG;
    return launch_cp_combine(s_loc, m, seq_seg, n_seqs, n_heads, s_start, final_state,
                             (cudaStream_t)stream);
}

int kda_cp_correct(const float *u, const float *s_start, const int32_t *cu_seg, int32_t n_seg,
                   const int32_t *skip_seg, int32_t n_skip, int64_t total_tokens, int32_t n_heads,
                   int32_t d, float *out, void *stream)
{
    const CallRange range("kda_cp_correct");
    if (n_seg < 0 || n_skip < 0 || total_tokens < 0 || n_heads < 1 || d < 1) return KDA_ERR_INVALID_ARG;
    if (d != 128) return KDA_ERR_UNSUPPORTED_SHAPE;
    if (n_seg > 0 && (!u || !s_start || !cu_seg || !out || (n_skip > 0 && !skip_seg)))
        return KDA_ERR_INVALID_ARG;
    const void *ptrs[] = {u, s_start, out};
    for (const void *p : ptrs)
        if (p && !aligned16(p)) return KDA_ERR_MISALIGNED;
    if ((reinterpret_cast<uintptr_t>(cu_seg) & 3u) != 0 || (reinterpret_cast<uintptr_t>(skip_seg) & 3u) != 0)
        return KDA_ERR_MISALIGNED;
    if (out && (out == u || reinterpret_cast<const void *>(out) == s_start)) return KDA_ERR_INVALID_ARG;
    return launch_cp_correct(u, s_start, cu_seg, n_seg, skip_seg, n_skip, n_heads, (long long)total_tokens,
                             out, (cudaStream_t)stream);
}

int64_t kda_prefill_staged_scratch(const int32_t *h_cu_seqlens, int32_t n_seqs, int64_t total_tokens,
                                   int64_t chunk_tokens)
{
    if (n_seqs < 0 || total_tokens < 0 || chunk_tokens < 1 || (n_seqs > 1 && !h_cu_seqlens)) return -1;
    return staged_scratch_ints(h_cu_seqlens, n_seqs, total_tokens, chunk_tokens);
}

int kda_prefill_staged(const void *h_q, const void *h_k, const void *h_v, const void *h_g,
                       const void *h_beta, const int32_t *h_cu_seqlens, int32_t n_seqs,
                       int64_t total_tokens, int32_t n_heads, int32_t dtype, int32_t out_dtype,
                       const float *init_state, void *d_q, void *d_k, void *d_v, void *d_g,
                       void *d_beta, void *d_out, void *h_out, float *final_state,
                       int32_t *d_scratch, int64_t scratch_ints, int64_t chunk_tokens, void *stream)
{
    const CallRange range("kda_prefill_staged");
    int rc = check_staged(h_q, h_k, h_v, h_g, h_beta, h_cu_seqlens, n_seqs, total_tokens, n_heads,
                          dtype, out_dtype, init_state, d_q, d_k, d_v, d_g, d_beta, d_out, h_out,
                          final_state, chunk_tokens);
    if (rc != KDA_OK) return rc;
    if (d_scratch && !aligned16(d_scratch)) return KDA_ERR_MISALIGNED;
    const int64_t need = staged_scratch_ints(h_cu_seqlens, n_seqs, total_tokens, chunk_tokens);
    if (need > 0 && (!d_scratch || scratch_ints < need)) return KDA_ERR_INVALID_ARG;
    const void *h_in[5] = {h_q, h_k, h_v, h_g, h_beta};
    void *d_in[5] = {d_q, d_k, d_v, d_g, d_beta};
    return run_prefill_staged(h_in, h_cu_seqlens, n_seqs, total_tokens, n_heads, dtype, out_dtype,
                              init_state, d_in, d_out, h_out, final_state, d_scratch, chunk_tokens,
                              (cudaStream_t)stream);
}

int kda_prefill_staged_static(const void *h_q, const void *h_k, const void *h_v, const void *h_g,
                              const void *h_beta, const int32_t *h_cu_seqlens, int32_t n_seqs,
                              int64_t total_tokens, int32_t n_heads, int32_t dtype, int32_t out_dtype,
                              const float *init_state, void *d_q, void *d_k, void *d_v, void *d_g,
                              void *d_beta, void *d_out, void *h_out, float *final_state,
                              int64_t chunk_tokens, void *stream)
{
    const CallRange range("kda_prefill_staged_static");
    int rc = check_staged(h_q, h_k, h_v, h_g, h_beta, h_cu_seqlens, n_seqs, total_tokens, n_heads,
                          dtype, out_dtype, init_state, d_q, d_k, d_v, d_g, d_beta, d_out, h_out,
                          final_state, chunk_tokens);
    if (rc != KDA_OK) return rc;
    const void *h_in[5] = {h_q, h_k, h_v, h_g, h_beta};
    void *d_in[5] = {d_q, d_k, d_v, d_g, d_beta};
    return run_prefill_staged_static(h_in, h_cu_seqlens, n_seqs, total_tokens, n_heads, dtype,
                                     out_dtype, init_state, d_in, d_out, h_out, final_state,
                                     chunk_tokens, (cudaStream_t)stream);
}

int kda_diag_device_timeout(int64_t timeout_cycles, void *stream)
{
    if (timeout_cycles < 1 || timeout_cycles > 4000000000LL) return KDA_ERR_INVALID_ARG;
    return kda::launch_wait_timeout_probe((long long)timeout_cycles, (cudaStream_t)stream);
}

int kda_diag_staged_handles(int64_t *created)
{
    if (!created) return KDA_ERR_INVALID_ARG;
    *created = staged_handles_created();
    return KDA_OK;
}

int kda_diag_bounds_check(int32_t run_probe, int32_t *site, void *stream)
{
    if (!site) return KDA_ERR_INVALID_ARG;
    if (run_probe && kda::launch_bounds_check_probe((cudaStream_t)stream) != KDA_OK) return KDA_ERR_CUDA;
    int32_t a = 0, b = 0;   // the default and the precise build of the tensor-core prefill
    if (kda::read_and_clear_debug_site((cudaStream_t)stream, &a) != KDA_OK ||
        kda::read_and_clear_debug_site_precise((cudaStream_t)stream, &b) != KDA_OK)
        return KDA_ERR_CUDA;
    *site = a != 0 ? a : b;
    return KDA_OK;
}

int kda_device_status(int32_t *status, void *stream)
{
    if (!status) return KDA_ERR_INVALID_ARG;
    int32_t a = 0, b = 0, c = 0;
    int rc = read_and_clear_status_state_copy((cudaStream_t)stream, &a);
    if (rc != KDA_OK) return rc;
    rc = read_and_clear_status_prefill_tc((cudaStream_t)stream, &b);
    if (rc != KDA_OK) return rc;
    int32_t bp = 0;
    rc = read_and_clear_status_prefill_tc_precise((cudaStream_t)stream, &bp);
    if (rc != KDA_OK) return rc;
    if (b == KDA_OK) b = bp;
    rc = read_and_clear_status_decode((cudaStream_t)stream, &c);
    if (rc != KDA_OK) return rc;
    int32_t cp = 0;
    rc = read_and_clear_status_cp((cudaStream_t)stream, &cp);
    if (rc != KDA_OK) return rc;
    if (c == KDA_OK) c = cp;
    *status = b != KDA_OK ? b : (c != KDA_OK ? c : a);
    return KDA_OK;
}

}  // extern "C"
