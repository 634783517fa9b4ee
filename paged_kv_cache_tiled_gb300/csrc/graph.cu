// A decode step captured once and replayed as a CUDA graph ("Fast Attention
// Kernels and Operator Fusion", section "Fusion and CUDA Graphs with
// torch.compile": a CUDA Graph records the sequence of GPU operations and
// replays it with one CPU submission, cutting launch overhead; replay needs
// stable memory addresses and compatible shapes, and suits repeated
// small-batch work such as decode).
//
// The step is the cache append of the new tokens followed by paged attention
// (the decode kernel and its merge, or the tensor-core path for longer
// chunks), captured from the same entry points a caller uses directly.  Those
// entry points never synchronise, allocate or read device memory on the host,
// so capturing them records exactly the launches an eager call makes.  Every
// pointer and size is fixed at capture; the caller changes the contents of
// the buffers (new q/k/v rows, slot mapping, block table, context lengths)
// between replays, and the kernels read them on the device.
#include <new>

#include "host_common.cuh"

struct fa_decode_graph {
    cudaGraph_t graph = nullptr;
    cudaGraphExec_t exec = nullptr;
    int launches = 0;
};

extern "C" {

fa_status fa_decode_graph_create(fa_decode_graph** out, const void* k_new, const void* v_new,
                                 const int32_t* slot_mapping, int n_new, fa_dtype in_dtype, const void* q,
                                 void* k_cache, void* v_cache, const int32_t* block_table, const int32_t* ctx_lens,
                                 const int32_t* q_lens, void* attn_out, int num_seqs, int max_blocks_per_seq,
                                 int num_blocks, int Hq, int Hkv, int d, int causal, float scale, int total_q,
                                 int max_q_len, void* ws, size_t ws_bytes) {
    using namespace fa;
    if (!out) return FA_ERR_INVALID_ARG;
    *out = nullptr;
    if (n_new < 0) return FA_ERR_INVALID_ARG;
    fa_status st = check_device();
    if (st != FA_OK) return st;
    cudaStream_t cap = nullptr;
    if (cudaStreamCreateWithFlags(&cap, cudaStreamNonBlocking) != cudaSuccess) return FA_ERR_CUDA;
    fa_decode_graph* g = new (std::nothrow) fa_decode_graph;
    if (!g) {
        cudaStreamDestroy(cap);
        return FA_ERR_CUDA;
    }
    // per-device setup (error word, tensor-map encoder, kernel attributes)
    // happens outside the capture, on the first eager-style query
    DevCtx ctx;
    if ((st = make_ctx(&ctx)) != FA_OK) {
        delete g;
        cudaStreamDestroy(cap);
        return st;
    }
    if (cudaStreamBeginCapture(cap, cudaStreamCaptureModeThreadLocal) != cudaSuccess) {
        delete g;
        cudaStreamDestroy(cap);
        return FA_ERR_CUDA;
    }
    int launches = 0;
    fa_stream_t s = reinterpret_cast<fa_stream_t>(cap);
    if (n_new > 0) {
        st = fa_cache_append(k_new, v_new, k_cache, v_cache, slot_mapping, n_new, Hkv, d, num_blocks, in_dtype, s);
        launches += fa_last_launch_count();
    }
    if (st == FA_OK) {
        st = fa_paged_attn(q, k_cache, v_cache, block_table, ctx_lens, q_lens, attn_out, num_seqs,
                           max_blocks_per_seq, num_blocks, Hq, Hkv, d, 16, causal, scale, total_q, max_q_len, ws,
                           ws_bytes, s);
        launches += fa_last_launch_count();
    }
    cudaGraph_t graph = nullptr;
    const cudaError_t ec = cudaStreamEndCapture(cap, &graph);
    cudaStreamDestroy(cap);
    if (st == FA_OK && (ec != cudaSuccess || !graph)) st = FA_ERR_CUDA;
    if (st == FA_OK && cudaGraphInstantiate(&g->exec, graph, 0) != cudaSuccess) st = FA_ERR_CUDA;
    if (st != FA_OK) {
        if (graph) cudaGraphDestroy(graph);
        delete g;
        set_launch_count(0);
        return st;
    }
    g->graph = graph;
    g->launches = launches;
    set_launch_count(0);  // nothing ran: capture only records
    *out = g;
    return FA_OK;
}

fa_status fa_decode_graph_launch(fa_decode_graph* g, fa_stream_t stream) {
    if (!g || !g->exec) return FA_ERR_INVALID_ARG;
    const fa_status st =
        cudaGraphLaunch(g->exec, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess ? FA_OK : FA_ERR_CUDA;
    fa::set_launch_count(st == FA_OK ? g->launches : 0);
    return st;
}

int fa_decode_graph_kernel_count(const fa_decode_graph* g) { return g ? g->launches : 0; }

void fa_decode_graph_destroy(fa_decode_graph* g) {
    if (!g) return;
    if (g->exec) cudaGraphExecDestroy(g->exec);
    if (g->graph) cudaGraphDestroy(g->graph);
    delete g;
}

}  // extern "C"
