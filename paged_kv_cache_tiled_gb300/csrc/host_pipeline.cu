// Prefill from and to host memory with the copies overlapped with the
// attention work.  The batch is split by sequence: while sequence b is
// computed on the caller's stream, the inputs of sequence b+1 are copied in on
// one internal stream and the output of sequence b-1 is copied out on
// another, so host-to-device copies, device-to-host copies and compute run at
// the same time.  Each sequence goes through fa_prefill unchanged (a batch of
// one), whose work units do not depend on the batch size, so the result is
// the one fa_prefill gives for the whole batch, bit for bit.
//
// The internal streams and events are created once per device and reused;
// a mutex keeps the enqueue of one call together.  Every stream/event
// operation is capturable, so a call may be recorded into a CUDA graph.
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

    // bytes of one sequence; d * 2 B is a multiple of 128, so every slice
    // keeps the 16-byte (inputs) and 32-byte (output) alignment
    const size_t q_b = (size_t)T * Hq * d * 2, kv_b = (size_t)T * Hkv * d * 2;
    auto at = [](const void* p, size_t off) { return static_cast<const char*>(p) + off; };
    auto atw = [](void* p, size_t off) { return static_cast<char*>(p) + off; };
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);

    HostPipe& hp = g_pipe[dev];
    std::lock_guard<std::mutex> lk(hp.mu);
    // events: fork, then per sequence "inputs copied" and "computed", then join
    if ((st = ensure_pipe(hp, 2 + 2 * (size_t)B)) != FA_OK) return st;
    cudaEvent_t fork = hp.ev[0], join = hp.ev[1];
    auto ok = [](cudaError_t e) { return e == cudaSuccess; };
    // the copies start after everything already queued on the caller's stream
    // (the device buffers may still be in use there)
    if (!ok(cudaEventRecord(fork, cs)) || !ok(cudaStreamWaitEvent(hp.in, fork, 0)) ||
        !ok(cudaStreamWaitEvent(hp.out, fork, 0)))
        return FA_ERR_CUDA;
    int launches = 0;
    for (int b = 0; b < B; ++b) {
        cudaEvent_t copied = hp.ev[2 + 2 * b], computed = hp.ev[3 + 2 * b];
        if (!ok(cudaMemcpyAsync(atw(q, b * q_b), at(q_host, b * q_b), q_b, cudaMemcpyHostToDevice, hp.in)) ||
            !ok(cudaMemcpyAsync(atw(k, b * kv_b), at(k_host, b * kv_b), kv_b, cudaMemcpyHostToDevice, hp.in)) ||
            !ok(cudaMemcpyAsync(atw(v, b * kv_b), at(v_host, b * kv_b), kv_b, cudaMemcpyHostToDevice, hp.in)) ||
            !ok(cudaEventRecord(copied, hp.in)) || !ok(cudaStreamWaitEvent(cs, copied, 0)))
            return FA_ERR_CUDA;
        st = fa_prefill(at(q, b * q_b), at(k, b * kv_b), at(v, b * kv_b), atw(out, b * q_b), 1, T, Hq, Hkv, d,
                        causal, scale, nullptr, stream);
        if (st != FA_OK) return st;
        launches += 1;
        if (!ok(cudaEventRecord(computed, cs)) || !ok(cudaStreamWaitEvent(hp.out, computed, 0)) ||
            !ok(cudaMemcpyAsync(atw(out_host, b * q_b), at(out, b * q_b), q_b, cudaMemcpyDeviceToHost, hp.out)))
            return FA_ERR_CUDA;
    }
    // later work on the caller's stream sees the output in host memory
    if (!ok(cudaEventRecord(join, hp.out)) || !ok(cudaStreamWaitEvent(cs, join, 0))) return FA_ERR_CUDA;
    set_launch_count(launches);
    return FA_OK;
}
