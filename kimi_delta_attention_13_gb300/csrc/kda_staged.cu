// kda_staged.cu -- prefill from pinned host memory with the copies overlapped with the compute.
//
// The packed tokens are cut into chunks.  Chunk c's inputs go host -> device on one internal
// stream, its prefill runs on the caller's stream once they have landed (every sequence resumes
// from its running state, kept in final_state: the recurrence hands the state from token to token,
// "Kimi K3 im Detail", section "Sequenz-Mixing: KDA-Zustand und globale MLA"), and its outputs go
// device -> host on a second internal stream.  Chunk c+1's upload therefore overlaps chunk c's
// prefill and chunk c-1's download, and both copy directions run at once.
//
// Downloads go by SM stores into the caller's pinned buffer when it is mapped into the device's
// address space (pinned host memory under unified addressing): on a GB300's host link, copy-engine
// uploads next to SM-store downloads moved 303 GB/s together, against 285 GB/s with copy engines in
// both directions.  Each direction alone runs at the same rate either way (211 GB/s up, 193 down).
#include <atomic>
#include <cstdint>
#include <mutex>
#include <vector>

#include "kda_internal.cuh"

namespace kda {
namespace {

// Sequence tables of kda_prefill_staged_static: a fixed device array instead of caller scratch.
// Calls share it, so each call's stream first waits for the previous call's last read of it.
constexpr int64_t kStaticTableInts = 1 << 20;
static __device__ __align__(256) int32_t g_staged_tables[kStaticTableInts];
std::mutex g_tables_mu;
constexpr int kMaxDevices = 64;
cudaEvent_t g_tables_free[kMaxDevices] = {};   // per device: recorded after the last call that read the table

// Streams and events of the staged calls, created on a device's first call and kept until the
// process exits: two non-blocking streams (uploads, downloads) and four events, reused by every
// later call on that device.  A call holds `mu` while it enqueues, so calls from several host
// threads take turns at enqueueing and share the two copy streams.
struct Resources {
    std::mutex mu;
    bool ready = false;
    cudaStream_t s_in = nullptr, s_out = nullptr;
    cudaEvent_t start = nullptr, done = nullptr, landed = nullptr, computed = nullptr;
};
Resources g_resources[kMaxDevices];
std::mutex g_resources_mu;
std::atomic<long long> g_handles_created{0};   // streams and events created by the staged calls

// The device that `stream` belongs to, which must be the current device (the kernels launch
// there).  KDA_ERR_INVALID_ARG for another device's stream.
int stream_device(cudaStream_t stream, int *dev)
{
    int cur = 0, sd = 0;
    if (cudaGetDevice(&cur) != cudaSuccess || cudaStreamGetDevice(stream, &sd) != cudaSuccess) return KDA_ERR_CUDA;
    if (sd != cur) return KDA_ERR_INVALID_ARG;
    if (cur < 0 || cur >= kMaxDevices) return KDA_ERR_CUDA;
    *dev = cur;
    return KDA_OK;
}

int device_resources(cudaStream_t stream, Resources **out)
{
    int dev = 0;
    const int rc = stream_device(stream, &dev);
    if (rc != KDA_OK) return rc;
    std::lock_guard<std::mutex> lock(g_resources_mu);
    Resources &r = g_resources[dev];
    if (!r.ready) {   // a set left partial by a failed creation is completed by the next call
        cudaStream_t *streams[2] = {&r.s_in, &r.s_out};
        cudaEvent_t *events[4] = {&r.start, &r.done, &r.landed, &r.computed};
        for (cudaStream_t *x : streams)
            if (!*x) {
                if (cudaStreamCreateWithFlags(x, cudaStreamNonBlocking) != cudaSuccess) {
                    *x = nullptr;
                    return KDA_ERR_CUDA;
                }
                ++g_handles_created;
            }
        for (cudaEvent_t *x : events)
            if (!*x) {
                if (cudaEventCreateWithFlags(x, cudaEventDisableTiming) != cudaSuccess) {
                    *x = nullptr;
                    return KDA_ERR_CUDA;
                }
                ++g_handles_created;
            }
        r.ready = true;
    }
    *out = &r;
    return KDA_OK;
}

// SM-store downloads: a few blocks fill the host link and leave most SMs to the next chunk's
// prefill (one whole SM per CTA).  On the T = 8192, H = 96 workload 64 blocks did slightly better
// than 32 and 16 (4.55, 4.57 and 4.59 ms per call).
constexpr int kStoreBlocks = 64;
constexpr int kStoreThreads = 512;

__global__ void __launch_bounds__(kStoreThreads) store_to_host_kernel(int4 *__restrict__ dst,
                                                                      const int4 *__restrict__ src,
                                                                      long long n16)
{
    const long long stride = (long long)gridDim.x * blockDim.x;
    long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x;
    for (; i + 3 * stride < n16; i += 4 * stride) {   // four loads in flight, then four stores
        const int4 a = src[i], b = src[i + stride], c = src[i + 2 * stride], d = src[i + 3 * stride];
        dst[i] = a;
        dst[i + stride] = b;
        dst[i + 2 * stride] = c;
        dst[i + 3 * stride] = d;
    }
    for (; i < n16; i += stride) dst[i] = src[i];
}

struct Chunk {
    long long t0, t1;   // token range
    int n_a, n_b;       // sequences n_a .. n_b (inclusive) intersect it
    int cu_off;         // its sub-batch cu table in the scratch (-1: one sequence, no table)
};

// Chunk boundaries: `chunk_tokens` tokens a chunk, except that the last chunk is cut in halves
// (whole multiples of 32 tokens when chunk_tokens is one) down to at most 128 tokens.  Once the
// last upload has landed, only the last piece's prefill and download remain, so the pipeline's
// drain is short.
std::vector<long long> bounds(long long T, long long chunk_tokens)
{
    std::vector<long long> b{0};
    long long t0 = 0;
    while (T - t0 > chunk_tokens) b.push_back(t0 += chunk_tokens);
    if (chunk_tokens % 32 == 0)
        while (T - t0 > 128) b.push_back(t0 += ((T - t0) / 2 + 31) / 32 * 32);
    if (T > t0) b.push_back(T);
    return b;
}

// The chunks and their sub-batch cu tables (appended to `tab`)
std::vector<Chunk> plan(const int32_t *cu, int n_seqs, long long T, long long chunk_tokens,
                        std::vector<int32_t> &tab)
{
    std::vector<Chunk> out;
    const std::vector<long long> b = bounds(T, chunk_tokens);
    int n = 0;
    for (size_t i = 0; i + 1 < b.size(); ++i) {
        const long long t0 = b[i], t1 = b[i + 1];
        while (n + 1 < n_seqs && cu[n + 1] <= t0) ++n;   // first sequence holding t0
        int m = n;
        while (m + 1 < n_seqs && cu[m + 1] < t1) ++m;    // last sequence holding a token < t1
        Chunk c{t0, t1, n, m, -1};
        if (m > n) {
            c.cu_off = (int)tab.size();
            tab.push_back(0);
            for (int s = n + 1; s <= m; ++s) tab.push_back((int32_t)(cu[s] - t0));
            tab.push_back((int32_t)(t1 - t0));
        }
        out.push_back(c);
    }
    return out;
}

}  // namespace

int64_t staged_scratch_ints(const int32_t *h_cu, int n_seqs, long long T, long long chunk_tokens)
{
    if (n_seqs <= 1 || T == 0) return 0;
    std::vector<int32_t> tab;
    plan(h_cu, n_seqs, T, chunk_tokens, tab);
    return (int64_t)tab.size();
}

int run_prefill_staged(const void *const h_in[5], const int32_t *h_cu, int n_seqs, long long T,
                       int H, int dtype, int out_dtype, const float *init_state, void *const d_in[5],
                       void *d_out, void *h_out, float *final_state, int32_t *d_scratch,
                       long long chunk_tokens, cudaStream_t stream)
{
    const size_t esz = dtype == KDA_BF16 ? 2 : 4, osz = out_dtype == KDA_BF16 ? 2 : 4;
    const size_t row = (size_t)H * 128;                       // elements of a token's q/k/v/g row
    const size_t blk = (size_t)H * 128 * 128 * sizeof(float);   // one sequence's states
    // the call's streams and events are the device's cached set, held for the whole enqueue
    Resources *res = nullptr;
    const int rdev = device_resources(stream, &res);
    if (rdev != KDA_OK) return rdev;
    std::lock_guard<std::mutex> lock(res->mu);
    // running states: the initial ones (or zeros), overwritten chunk by chunk
    cudaError_t e = cudaSuccess;
    if (!init_state)
        e = cudaMemsetAsync(final_state, 0, blk * n_seqs, stream);
    else if (init_state != final_state)
        e = cudaMemcpyAsync(final_state, init_state, blk * n_seqs, cudaMemcpyDeviceToDevice, stream);
    if (e != cudaSuccess) return KDA_ERR_CUDA;
    if (T == 0) return KDA_OK;
    std::vector<int32_t> tab;
    const std::vector<Chunk> chunks = plan(h_cu, n_seqs, T, chunk_tokens, tab);
    if (!tab.empty() &&   // pageable source: the call returns once the table has been taken
        cudaMemcpyAsync(d_scratch, tab.data(), tab.size() * sizeof(int32_t), cudaMemcpyHostToDevice,
                        stream) != cudaSuccess)
        return KDA_ERR_CUDA;

    // the device's view of h_out for SM-store downloads (nullptr: copy-engine downloads)
    char *h_out_dev = nullptr;
    if (((uintptr_t)h_out | (uintptr_t)d_out) % 16 == 0 &&
        cudaHostGetDevicePointer(reinterpret_cast<void **>(&h_out_dev), h_out, 0) != cudaSuccess) {
        h_out_dev = nullptr;
        (void)cudaGetLastError();   // pageable or unregistered memory: not an error here
    }

    int rc = KDA_OK;
    auto ok = [&](cudaError_t x) {
        if (x != cudaSuccess && rc == KDA_OK) rc = KDA_ERR_CUDA;
        return rc == KDA_OK;
    };
    ok(cudaEventRecord(res->start, stream));
    ok(cudaStreamWaitEvent(res->s_in, res->start, 0));
    ok(cudaStreamWaitEvent(res->s_out, res->start, 0));
    for (size_t i = 0; rc == KDA_OK && i < chunks.size(); ++i) {
        const Chunk &c = chunks[i];
        const size_t rows = (size_t)(c.t1 - c.t0);
        // inputs of the chunk: q, k, v, g rows, then beta
        for (int x = 0; x < 5 && rc == KDA_OK; ++x) {
            const size_t w = (x < 4 ? row : (size_t)H) * esz;
            ok(cudaMemcpyAsync(static_cast<char *>(d_in[x]) + c.t0 * w, static_cast<const char *>(h_in[x]) + c.t0 * w,
                               rows * w, cudaMemcpyHostToDevice, res->s_in));
        }
        // a wait takes the event as last recorded, so one event serves every chunk
        ok(cudaEventRecord(res->landed, res->s_in));
        ok(cudaStreamWaitEvent(stream, res->landed, 0));
        if (rc == KDA_OK) {
            const int n_sub = c.n_b - c.n_a + 1;
            void *p[5];
            for (int x = 0; x < 5; ++x)
                p[x] = static_cast<char *>(d_in[x]) + c.t0 * (x < 4 ? row : (size_t)H) * esz;
            float *st = final_state + (size_t)c.n_a * H * 128 * 128;
            const int r = kda_prefill(p[0], p[1], p[2], p[3], p[4],
                                      c.cu_off < 0 ? nullptr : d_scratch + c.cu_off, n_sub,
                                      (int64_t)rows, H, 128, 128, dtype, out_dtype, st,
                                      static_cast<char *>(d_out) + c.t0 * row * osz, st, 0, nullptr,
                                      stream);
            if (r != KDA_OK) rc = r;
        }
        ok(cudaEventRecord(res->computed, stream));
        ok(cudaStreamWaitEvent(res->s_out, res->computed, 0));
        const size_t off = c.t0 * row * osz, bytes = rows * row * osz;   // multiples of 256 B
        if (h_out_dev) {
            store_to_host_kernel<<<kStoreBlocks, kStoreThreads, 0, res->s_out>>>(
                reinterpret_cast<int4 *>(h_out_dev + off),
                reinterpret_cast<const int4 *>(static_cast<const char *>(d_out) + off),
                (long long)(bytes / 16));
            ok(cudaGetLastError());
        } else {
            ok(cudaMemcpyAsync(static_cast<char *>(h_out) + off, static_cast<const char *>(d_out) + off,
                               bytes, cudaMemcpyDeviceToHost, res->s_out));
        }
    }
    // the caller's stream continues after the last download (also after an error, so that no
    // later work of the caller overtakes copies already queued)
    cudaEventRecord(res->done, res->s_out);
    cudaStreamWaitEvent(stream, res->done, 0);
    return rc;
}

int run_prefill_staged_static(const void *const h_in[5], const int32_t *h_cu, int n_seqs, long long T,
                              int H, int dtype, int out_dtype, const float *init_state,
                              void *const d_in[5], void *d_out, void *h_out, float *final_state,
                              long long chunk_tokens, cudaStream_t stream)
{
    if (staged_scratch_ints(h_cu, n_seqs, T, chunk_tokens) > kStaticTableInts) return KDA_ERR_INVALID_ARG;
    int dev = 0;
    const int sd = stream_device(stream, &dev);   // the array and event of the stream's device
    if (sd != KDA_OK) return sd;
    void *tables = nullptr;
    if (cudaGetSymbolAddress(&tables, g_staged_tables) != cudaSuccess) return KDA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_tables_mu);
    cudaEvent_t &free_ev = g_tables_free[dev];
    if (!free_ev) {
        if (cudaEventCreateWithFlags(&free_ev, cudaEventDisableTiming) != cudaSuccess) {
            free_ev = nullptr;
            return KDA_ERR_CUDA;
        }
        ++g_handles_created;
    }
    // the table upload below is ordered after the previous call's prefills (a fresh event counts
    // as complete)
    if (cudaStreamWaitEvent(stream, free_ev, 0) != cudaSuccess) return KDA_ERR_CUDA;
    const int rc = run_prefill_staged(h_in, h_cu, n_seqs, T, H, dtype, out_dtype, init_state, d_in,
                                      d_out, h_out, final_state, static_cast<int32_t *>(tables),
                                      chunk_tokens, stream);
    // `stream` is ordered after this call's last prefill (and download)
    if (cudaEventRecord(free_ev, stream) != cudaSuccess && rc == KDA_OK) return KDA_ERR_CUDA;
    return rc;
}

long long staged_handles_created() { return g_handles_created.load(); }

}  // namespace kda
