// Prefill from and to host memory with the copies overlapped with the
// attention work.  The key and value rows go in first (one copy each); then
// the query rows of every sequence in row chunks -- chunk c is rows
// [c*R, (c+1)*R) -- from the last chunk to the first.  Chunk c's attention
// runs on the caller's stream as soon as its query rows are in, and its output
// goes out on a second internal stream, so host-to-device copies, compute and
// device-to-host copies overlap at the grain of a chunk.  Going from the last
// rows to the first puts the chunks with the most keys to see (under a causal
// mask, "FlashAttention-Style Kernels": a query tile is combined only with the
// key tiles it can see) early, behind copies still to come, and leaves the
// cheapest chunk for the end, where nothing else is left to hide it.  Each
// chunk's launch computes the same query tiles against the same key tiles in
// the same order as fa_prefill over the whole batch, so the output equals that
// call's bit for bit.
//
// The internal streams and events are created once per device and reused;
// a mutex keeps the enqueue of one call together.  Every stream/event
// operation is capturable, so a call may be recorded into a CUDA graph.
#include <algorithm>
#include <cmath>
#include <mutex>
#include <vector>

#include "host_common.cuh"

namespace fa {
namespace {

constexpr int kMaxPipeDevices = 64;

struct HostPipe {
    std::mutex mu;
    cudaStream_t in = nullptr, out = nullptr;  // host-to-device, device-to-host
    std::vector<cudaEvent_t> ev;                // reused event pool
};
HostPipe g_pipe[kMaxPipeDevices];

// Grows the event pool of `hp` to at least n events (call under hp.mu).
fa_status ensure_pipe(HostPipe& hp, size_t n) {
    if (!hp.in && cudaStreamCreateWithFlags(&hp.in, cudaStreamNonBlocking) != cudaSuccess) return FA_ERR_CUDA;
    if (!hp.out && cudaStreamCreateWithFlags(&hp.out, cudaStreamNonBlocking) != cudaSuccess) return FA_ERR_CUDA;
    while (hp.ev.size() < n) {
        cudaEvent_t e = nullptr;
        if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) return FA_ERR_CUDA;
        hp.ev.push_back(e);
    }
    return FA_OK;
}

}  // namespace
}  // namespace fa

using namespace fa;

extern "C" fa_status fa_prefill_host(const void* q_host, const void* k_host, const void* v_host, void* out_host,
                                     void* q, void* k, void* v, void* out, int B, int T, int Hq, int Hkv, int d,
                                     int causal, float scale, fa_stream_t stream) {
    set_launch_count(0);
    if (B < 0 || T < 0 || Hq <= 0 || Hkv <= 0 || !(scale > 0.f) || !std::isfinite(scale)) return FA_ERR_INVALID_ARG;
    if ((d != 64 && d != 128) || Hq % Hkv != 0) return FA_ERR_UNSUPPORTED;
    if (B == 0 || T == 0) return FA_OK;
    if (!q_host || !k_host || !v_host || !out_host || !q || !k || !v || !out) return FA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned32(out)) return FA_ERR_INVALID_ARG;
    fa_status st = check_device();
    if (st != FA_OK) return st;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxPipeDevices) return FA_ERR_CUDA;

    // Row chunks: a multiple of 128 rows, about T/4 (each chunk costs one copy
    // in, one launch and one copy out; finer chunks lose more to those fixed
    // costs than they gain in overlap); d * 2 B is a multiple of 128, so every
    // slice keeps the 16-byte (inputs) and 32-byte (output) alignment.
    const int R = std::max(128, (T / 4 + 127) / 128 * 128);
    const int nchunks = (T + R - 1) / R;
    const size_t qrow = (size_t)Hq * d * 2, kvrow = (size_t)Hkv * d * 2;  // bytes of one row
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    auto ok = [](cudaError_t e) { return e == cudaSuccess; };
    // rows [r0, r0 + n) of every sequence: B slices, T rows apart
    auto copy_rows = [&](void* dst, const void* src, size_t row_bytes, int r0, int n, cudaMemcpyKind kind,
                         cudaStream_t st) {
        const size_t pitch = (size_t)T * row_bytes;
        return ok(cudaMemcpy2DAsync(static_cast<char*>(dst) + r0 * row_bytes, pitch,
                                    static_cast<const char*>(src) + r0 * row_bytes, pitch, (size_t)n * row_bytes, B,
                                    kind, st));
    };

    HostPipe& hp = g_pipe[dev];
    std::lock_guard<std::mutex> lk(hp.mu);
    // events: fork, join, then per chunk "query rows copied" and "computed"
    if ((st = ensure_pipe(hp, 2 + 2 * (size_t)nchunks)) != FA_OK) return st;
    cudaEvent_t fork = hp.ev[0], join = hp.ev[1];
    // the copies start after everything already queued on the caller's stream
    // (the device buffers may still be in use there)
    if (!ok(cudaEventRecord(fork, cs)) || !ok(cudaStreamWaitEvent(hp.in, fork, 0)) ||
        !ok(cudaStreamWaitEvent(hp.out, fork, 0)))
        return FA_ERR_CUDA;
    const size_t kv_bytes = (size_t)B * T * kvrow;
    if (!ok(cudaMemcpyAsync(k, k_host, kv_bytes, cudaMemcpyHostToDevice, hp.in)) ||
        !ok(cudaMemcpyAsync(v, v_host, kv_bytes, cudaMemcpyHostToDevice, hp.in)))
        return FA_ERR_CUDA;
    for (int c = nchunks - 1; c >= 0; --c) {
        const int r0 = c * R, n = std::min(R, T - r0);
        if (!copy_rows(q, q_host, qrow, r0, n, cudaMemcpyHostToDevice, hp.in) ||
            !ok(cudaEventRecord(hp.ev[2 + 2 * c], hp.in)))
            return FA_ERR_CUDA;
    }
    int launches = 0;
    for (int c = nchunks - 1; c >= 0; --c) {
        const int r0 = c * R, n = std::min(R, T - r0);
        cudaEvent_t copied = hp.ev[2 + 2 * c], computed = hp.ev[3 + 2 * c];
        if (!ok(cudaStreamWaitEvent(cs, copied, 0))) return FA_ERR_CUDA;
        st = launch_prefill_rows(q, k, v, out, B, T, Hq, Hkv, d, causal, scale, r0, n, causal ? r0 + n : T, cs);
        if (st != FA_OK) return st;
        ++launches;
        if (!ok(cudaEventRecord(computed, cs)) || !ok(cudaStreamWaitEvent(hp.out, computed, 0)) ||
            !copy_rows(out_host, out, qrow, r0, n, cudaMemcpyDeviceToHost, hp.out))
            return FA_ERR_CUDA;
    }
    // later work on the caller's stream sees the output in host memory
    if (!ok(cudaEventRecord(join, hp.out)) || !ok(cudaStreamWaitEvent(cs, join, 0))) return FA_ERR_CUDA;
    set_launch_count(launches);
    return FA_OK;
}
