// Paged attention ("Fast Attention Kernels and Operator Fusion", section
// "Paged Attention Kernels"): keys and values sit in 16-token blocks of a
// shared pool, [num_blocks, Hkv, 16, d] bf16, and every access goes through
// the per-sequence block table ("the kernel cannot assume that K[t+1] is
// adjacent to K[t]").
//
// Decode rows (the section "FlashAttention-Style Kernels" notes that decode
// has one or a few queries and is dominated by reading the growing cache)
// take a bandwidth-bound split-KV kernel:
//   * one CTA per (sequence, kv head, split of `split_blocks` blocks); its four
//     warps take every fourth block of the split;
//   * each warp streams its blocks through a private 3-stage ring of shared
//     memory with TMA (one 2 KB box per 64 channels of K and of V, 128-byte
//     swizzled so the fragment loads below are bank-conflict free); the
//     physical block id is read from the block table just before the copy;
//   * all Hq/Hkv query heads of the kv head (times the chunk's query tokens,
//     at most 16 rows) share each K/V load: they form the M dimension of
//     m16n8k16 warp MMAs, so K and V are read from HBM exactly once;
//   * the running row max / row sum are kept in fp32 (online softmax with
//     base-2 exponentials, scale * log2(e) folded into the scores);
//   * the four warps' states are merged in shared memory; a single split
//     writes the final bf16 output, several splits write fp32 partials
//     (unnormalised O, running max, running sum) merged by a second kernel
//     with log-sum-exp weights.
// Longer chunks take the tensor-core kernel (attn_tc.cu) through a work list
// built on the device by `paged_meta_kernel`.
#include <cstdlib>
#include <mutex>

#include "host_common.cuh"

namespace fa {

constexpr int kBS = 16;            // tokens per block
constexpr int kDecodeWarps = 4;    // warps per decode CTA
constexpr int kDecodeStages = 3;   // ring depth per warp
constexpr int kDecodeRows = 16;    // M of the warp MMA

// Launched from attn_tc.cu.
fa_status launch_paged_prefill(const void* q, const void* k_cache, const void* v_cache, const int32_t* block_table,
                               const int32_t* ctx_lens, const int32_t* q_lens, const int32_t* q_start,
                               const int32_t* work_list, const int32_t* work_count, void* out, int num_seqs,
                               int mbps, int num_blocks, int Hq, int Hkv, int d, int causal, float scale,
                               int total_q, cudaStream_t s, const DevCtx& ctx);

__host__ __device__ inline bool is_decode_row(int q_len, int g) { return q_len >= 1 && g * q_len <= kDecodeRows; }

// ------------------------------------------------------------------ layout --
struct PagedWs {
    size_t q_start, work_count, work_list, part_o, part_ml, total;
    int split_blocks, max_splits, max_entries;
};

// Blocks per decode split (per CTA).  FA_DECODE_SPLIT_BLOCKS (8..256) overrides
// the default for tuning; the workspace size query uses the same value.
inline int decode_split_blocks(int mbps) {
    (void)mbps;
    static const int v = [] {
        const char* e = getenv("FA_DECODE_SPLIT_BLOCKS");
        const int x = e ? atoi(e) : 0;
        return (x >= 8 && x <= 256) ? x : 64;
    }();
    return v;
}

inline PagedWs paged_ws_layout(int num_seqs, int mbps, int Hq, int Hkv, int d, int total_q) {
    (void)Hq;
    PagedWs w{};
    w.split_blocks = decode_split_blocks(mbps);
    w.max_splits = (mbps + w.split_blocks - 1) / w.split_blocks;
    if (w.max_splits < 1) w.max_splits = 1;
    w.max_entries = total_q / 128 + num_seqs + 1;
    size_t off = 0;
    w.q_start = off;
    off = align256(off + sizeof(int32_t) * (size_t)(num_seqs + 1));
    w.work_count = off;
    off = align256(off + sizeof(int32_t) * 4);
    w.work_list = off;
    off = align256(off + sizeof(int32_t) * 2 * (size_t)w.max_entries);
    w.part_o = off;
    off = align256(off + sizeof(float) * (size_t)num_seqs * Hkv * w.max_splits * kDecodeRows * d);
    w.part_ml = off;
    off = align256(off + sizeof(float2) * (size_t)num_seqs * Hkv * w.max_splits * kDecodeRows);
    w.total = off;
    return w;
}

// Sum of q_lens[0..s) by the whole CTA (blockDim.x threads, multiple of 32).
__device__ int cta_prefix(const int32_t* __restrict__ q_lens, int s, int* red) {
    int acc = 0;
    for (int i = threadIdx.x; i < s; i += blockDim.x) acc += __ldg(q_lens + i);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    const int w = threadIdx.x >> 5, nw = blockDim.x >> 5;
    __syncthreads();
    if ((threadIdx.x & 31) == 0) red[w] = acc;
    __syncthreads();
    int tot = 0;
    for (int i = 0; i < nw; ++i) tot += red[i];
    __syncthreads();
    return tot;
}

// -------------------------------------------------------------- decode -----
template <int D>
struct DecodeSmem {
    static constexpr int kPage = kBS * D * 2;                      // bytes of one K (or V) page
    static constexpr int kStage = 2 * kPage;                       // K page + V page
    static constexpr int kRing = kDecodeWarps * kDecodeStages * kStage;
    static constexpr int kCombine = kDecodeWarps * kDecodeRows * (D + 2) * 4;
    static constexpr int kData = kRing > kCombine ? kRing : kCombine;
    static constexpr int kBytes = 1024 /*align slack*/ + kData + (kDecodeWarps * kDecodeStages + 1) * 8 + 64;
};

template <int D>
__global__ void __launch_bounds__(kDecodeWarps * 32, 2)
    paged_decode_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                        const uint16_t* __restrict__ q, const int32_t* __restrict__ bt,
                        const int32_t* __restrict__ ctx_lens, const int32_t* __restrict__ q_lens,
                        uint16_t* __restrict__ out, float* __restrict__ part_o, float2* __restrict__ part_ml,
                        int mbps, int num_blocks, int Hq, int Hkv, int causal, float scale_log2, int split_blocks,
                        int max_splits, DevCtx ctx) {
    using L = DecodeSmem<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kData);
    uint64_t* never = bars + kDecodeWarps * kDecodeStages;  // nothing arrives on it (time-out test hook)
    int* red = reinterpret_cast<int*>(never + 1);
    volatile int* abort_flag = red + 8;

    // the merge kernel that follows may be scheduled now; it waits for this
    // grid's completion before reading anything
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int sp = blockIdx.x, hk = blockIdx.y, s = blockIdx.z;
    const int g = Hq / Hkv;
    const int q_len = __ldg(q_lens + s), ctx_len = __ldg(ctx_lens + s);
    if (!is_decode_row(q_len, g)) return;
    if (q_len > ctx_len || ctx_len > mbps * kBS) {
        if (sp == 0 && hk == 0 && threadIdx.x == 0) raise_error(ctx, ERR_BOUNDS_BIT);
        return;
    }
    const int nblk = (ctx_len + kBS - 1) / kBS;
    const int nsplit = (nblk + split_blocks - 1) / split_blocks;
    if (sp >= nsplit) return;
    const int blk0 = sp * split_blocks, blk1 = min(nblk, blk0 + split_blocks);
    const int nrows = g * q_len;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int i = 0; i < kDecodeWarps * kDecodeStages + 1; ++i) mbar_init(&bars[i], 1);
        *abort_flag = 0;
        mbar_fence_init();
    }
    __syncthreads();

    uint8_t* ring = smem + warp * kDecodeStages * L::kStage;
    uint64_t* wbar = bars + warp * kDecodeStages;
    const int n_mine = (blk1 - blk0 - warp + kDecodeWarps - 1) / kDecodeWarps;  // blocks blk0+warp+4i

    auto issue = [&](int i) {
        const int stage = i % kDecodeStages;
        const int lb = blk0 + warp + kDecodeWarps * i;
        int phys = __ldg(bt + (long)s * mbps + lb);
        if (phys < 0 || phys >= num_blocks) {
            raise_error(ctx, ERR_BOUNDS_BIT);
            phys = num_blocks;  // outside the tensor map: the copy fills zeros
        }
        uint8_t* kp = ring + stage * L::kStage;
        uint8_t* vp = kp + L::kPage;
        mbar_arrive_expect_tx(&wbar[stage], L::kStage);
#pragma unroll
        for (int h = 0; h < D / 64; ++h) {
            tma_load_4d(kp + h * 2048, &tm_k, &wbar[stage], h * 64, 0, hk, phys);
            tma_load_4d(vp + h * 2048, &tm_v, &wbar[stage], h * 64, 0, hk, phys);
        }
    };
    bool ok = !ctx.force_timeout || mbar_wait_warp(never, 0, ctx.wait_ns, abort_flag);
    if (!ok && lane == 0) {
        raise_error(ctx, ERR_TIMEOUT_BIT);
        *abort_flag = 1;
    }
    int issued = 0;  // lane 0's count of copies issued
    if (lane == 0 && ok)
        for (; issued < n_mine && issued < kDecodeStages; ++issued) issue(issued);
    // the first copies are in flight; the query offset is computed meanwhile
    const int q0 = cta_prefix(q_lens, s, red);

    // Q fragments (A operand, rows r = token * g + head-in-group)
    const int gid = lane >> 2, tig = lane & 3;
    uint32_t qa[D / 16][4];
    {
        const int rows_[2] = {gid, gid + 8};
        const uint16_t* qrow[2];
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const int r = rows_[i];
            qrow[i] = r < nrows ? q + ((long)(q0 + r / g) * Hq + hk * g + r % g) * D : nullptr;
        }
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
            const int c = ks * 16 + tig * 2;
            qa[ks][0] = qrow[0] ? __ldg(reinterpret_cast<const uint32_t*>(qrow[0] + c)) : 0u;
            qa[ks][1] = qrow[1] ? __ldg(reinterpret_cast<const uint32_t*>(qrow[1] + c)) : 0u;
            qa[ks][2] = qrow[0] ? __ldg(reinterpret_cast<const uint32_t*>(qrow[0] + c + 8)) : 0u;
            qa[ks][3] = qrow[1] ? __ldg(reinterpret_cast<const uint32_t*>(qrow[1] + c + 8)) : 0u;
        }
    }
    // causal limit per fragment row: keys <= pos(row) are visible
    const int pos_r0 = causal ? ctx_len - q_len + gid / g : ctx_len - 1;
    const int pos_r1 = causal ? ctx_len - q_len + (gid + 8) / g : ctx_len - 1;

    float o[D / 8][4];
#pragma unroll
    for (int n = 0; n < D / 8; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;

    const int mi = lane >> 3, r8 = lane & 7;
    int consumed = 0;
    for (int i = 0; ok && i < n_mine; ++i, consumed = i) {
        const int stage = i % kDecodeStages;
        if (!mbar_wait_warp(&wbar[stage], (i / kDecodeStages) & 1, ctx.wait_ns, abort_flag)) {
            if (lane == 0) {
                raise_error(ctx, ERR_TIMEOUT_BIT);
                *abort_flag = 1;
            }
            ok = false;
            break;
        }
        const uint32_t kbase = smem_u32(ring + stage * L::kStage);
        const uint32_t vbase = kbase + L::kPage;
        const int lb = blk0 + warp + kDecodeWarps * i;
        const int tok0 = lb * kBS;

        // S = Q K^T : 16 rows x 16 tokens
        float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
            const int tok = (mi >> 1) * 8 + r8;
            const int chunk = ks * 2 + (mi & 1);
            uint32_t b0, b1, b2, b3;
            ldsm_x4(kbase + (chunk >> 3) * 2048 + sw128_offset(tok, chunk & 7), b0, b1, b2, b3);
            mma_bf16_16816(sc[0], qa[ks], b0, b1);
            mma_bf16_16816(sc[1], qa[ks], b2, b3);
        }
        // mask + online softmax (base 2)
        float x[2][4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int t = tok0 + nt * 8 + tig * 2 + (e & 1);
                const int lim = (e < 2) ? pos_r0 : pos_r1;
                x[nt][e] = (t <= lim && t < ctx_len) ? sc[nt][e] * scale_log2 : -INFINITY;
            }
        float mx0 = fmaxf(fmaxf(x[0][0], x[0][1]), fmaxf(x[1][0], x[1][1]));
        float mx1 = fmaxf(fmaxf(x[0][2], x[0][3]), fmaxf(x[1][2], x[1][3]));
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
        const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
        const float mu0 = mn0 == -INFINITY ? 0.f : mn0, mu1 = mn1 == -INFINITY ? 0.f : mn1;
        const float a0 = fast_exp2(m0 - mu0), a1 = fast_exp2(m1 - mu1);
        m0 = mn0;
        m1 = mn1;
        float p[2][4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            p[nt][0] = fast_exp2(x[nt][0] - mu0);
            p[nt][1] = fast_exp2(x[nt][1] - mu0);
            p[nt][2] = fast_exp2(x[nt][2] - mu1);
            p[nt][3] = fast_exp2(x[nt][3] - mu1);
        }
        l0 = l0 * a0 + (p[0][0] + p[0][1] + p[1][0] + p[1][1]);
        l1 = l1 * a1 + (p[0][2] + p[0][3] + p[1][2] + p[1][3]);
        if (__any_sync(0xffffffffu, a0 != 1.f || a1 != 1.f)) {
#pragma unroll
            for (int n = 0; n < D / 8; ++n) {
                o[n][0] *= a0;
                o[n][1] *= a0;
                o[n][2] *= a1;
                o[n][3] *= a1;
            }
        }
        uint32_t pa[4] = {pack_bf16x2(p[0][0], p[0][1]), pack_bf16x2(p[0][2], p[0][3]),
                          pack_bf16x2(p[1][0], p[1][1]), pack_bf16x2(p[1][2], p[1][3])};
        // O += P V : V rows past the context are zeroed so stale cache words
        // (possibly NaN) cannot reach the accumulator through a zero weight
        const int nvalid = ctx_len - tok0;  // >= 1
        const uint32_t zlo0 = (tig * 2 < nvalid ? 0x0000ffffu : 0u) | (tig * 2 + 1 < nvalid ? 0xffff0000u : 0u);
        const uint32_t zhi0 =
            (tig * 2 + 8 < nvalid ? 0x0000ffffu : 0u) | (tig * 2 + 9 < nvalid ? 0xffff0000u : 0u);
#pragma unroll
        for (int dn = 0; dn < D / 16; ++dn) {
            const int tok = (mi & 1) * 8 + r8;
            const int chunk = dn * 2 + (mi >> 1);
            uint32_t b0, b1, b2, b3;
            ldsm_x4_t(vbase + (chunk >> 3) * 2048 + sw128_offset(tok, chunk & 7), b0, b1, b2, b3);
            b0 &= zlo0;
            b2 &= zlo0;
            b1 &= zhi0;
            b3 &= zhi0;
            mma_bf16_16816(o[2 * dn], pa, b0, b1);
            mma_bf16_16816(o[2 * dn + 1], pa, b2, b3);
        }
        __syncwarp();
        if (lane == 0 && issued < n_mine) issue(issued++);
    }
    if (!ok && lane == 0) {
        // drain: let the copies this warp issued but did not consume land
        // before the CTA can exit
        for (int i = consumed; i < issued; ++i)
            (void)mbar_wait_bounded(&wbar[i % kDecodeStages], (i / kDecodeStages) & 1, 1000000000ull, nullptr);
    }
    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);

    __syncthreads();  // ring no longer read; reuse it for the cross-warp merge
    if (*abort_flag) return;
    float* ow = reinterpret_cast<float*>(smem);                       // [warp][row][D]
    float* mlw = ow + kDecodeWarps * kDecodeRows * D;                  // [warp][row][2]
#pragma unroll
    for (int n = 0; n < D / 8; ++n) {
        const int c = n * 8 + tig * 2;
        ow[(warp * kDecodeRows + gid) * D + c] = o[n][0];
        ow[(warp * kDecodeRows + gid) * D + c + 1] = o[n][1];
        ow[(warp * kDecodeRows + gid + 8) * D + c] = o[n][2];
        ow[(warp * kDecodeRows + gid + 8) * D + c + 1] = o[n][3];
    }
    if (tig == 0) {
        mlw[(warp * kDecodeRows + gid) * 2] = m0;
        mlw[(warp * kDecodeRows + gid) * 2 + 1] = l0;
        mlw[(warp * kDecodeRows + gid + 8) * 2] = m1;
        mlw[(warp * kDecodeRows + gid + 8) * 2 + 1] = l1;
    }
    __syncthreads();
    const int per = blockDim.x / D > 0 ? blockDim.x / D : 1;  // threads per column group
    const int c = threadIdx.x % D;
    for (int r = threadIdx.x / D; r < nrows; r += per) {
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kDecodeWarps; ++w) M = fmaxf(M, mlw[(w * kDecodeRows + r) * 2]);
        float acc = 0.f, lsum = 0.f;
        if (M != -INFINITY) {
#pragma unroll
            for (int w = 0; w < kDecodeWarps; ++w) {
                const float a = fast_exp2(mlw[(w * kDecodeRows + r) * 2] - M);
                acc += a * ow[(w * kDecodeRows + r) * D + c];
                lsum += a * mlw[(w * kDecodeRows + r) * 2 + 1];
            }
        }
        if (nsplit == 1) {
            const float val = lsum > 0.f ? acc / lsum : 0.f;
            __nv_bfloat16 b = __float2bfloat16_rn(val);
            out[((long)(q0 + r / g) * Hq + hk * g + r % g) * D + c] = *reinterpret_cast<uint16_t*>(&b);
        } else {
            const long slot = (((long)s * Hkv + hk) * max_splits + sp) * kDecodeRows + r;
            part_o[slot * D + c] = acc;
            if (c == 0) part_ml[slot] = make_float2(M, lsum);
        }
    }
}

// Merges split partials: m = max_s m_s, l = sum_s 2^(m_s - m) l_s,
// O = sum_s 2^(m_s - m) O_s / l  (O_s unnormalised, all in base 2).
// One warp per row (8 warps, rows strided), lane j owns channels 4j..4j+3 and
// split j's statistics, so every load of a row is issued at once.  Launched as
// a programmatic dependent of the decode kernel: it may start early and waits
// for that grid's results with griddepcontrol.wait.
constexpr int kMergeThreads = 256;
template <int D>
__global__ void __launch_bounds__(kMergeThreads) paged_merge_kernel(const int32_t* __restrict__ ctx_lens,
                                                                    const int32_t* __restrict__ q_lens,
                                                                    const float* __restrict__ part_o,
                                                                    const float2* __restrict__ part_ml,
                                                                    uint16_t* __restrict__ out, int Hq, int Hkv,
                                                                    int split_blocks, int max_splits, int mbps) {
    __shared__ int red[kMergeThreads / 32];
    const int s = blockIdx.x, hk = blockIdx.y, g = Hq / Hkv;
    const int q_len = __ldg(q_lens + s), ctx_len = __ldg(ctx_lens + s);
    const bool active = is_decode_row(q_len, g) && q_len <= ctx_len && ctx_len <= mbps * kBS;
    const int nblk = (ctx_len + kBS - 1) / kBS;
    const int nsplit = (nblk + split_blocks - 1) / split_blocks;
    if (!active || nsplit <= 1) {
        // even a CTA with nothing to do waits for the decode grid, so this grid
        // never completes ahead of the one it depends on
        asm volatile("griddepcontrol.wait;" ::: "memory");
        return;
    }
    const int q0 = cta_prefix(q_lens, s, red);  // inputs only: no need to wait for the decode grid yet
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int nrows = g * q_len;
    const long base = ((long)s * Hkv + hk) * max_splits;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    constexpr int kPer = D / 32;  // channels per lane
    for (int r = warp; r < nrows; r += kMergeThreads / 32) {
        float M = -INFINITY;
        for (int s0 = lane; s0 < nsplit; s0 += 32) M = fmaxf(M, part_ml[(base + s0) * kDecodeRows + r].x);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
        float acc[kPer];
#pragma unroll
        for (int c = 0; c < kPer; ++c) acc[c] = 0.f;
        float lsum = 0.f;
        if (M != -INFINITY) {
            for (int c0 = 0; c0 < nsplit; c0 += 32) {
                float w = 0.f;
                if (c0 + lane < nsplit) {
                    const float2 ml = part_ml[(base + c0 + lane) * kDecodeRows + r];
                    w = fast_exp2(ml.x - M);
                    lsum += w * ml.y;
                }
                const int n = min(32, nsplit - c0);
                const float* src0 = part_o + ((base + c0) * kDecodeRows + r) * D + lane * kPer;
                const long stride = (long)kDecodeRows * D;  // floats between consecutive splits
                int j = 0;
                for (; j + 4 <= n; j += 4) {  // four splits' loads in flight at once
                    float v[4][kPer];
#pragma unroll
                    for (int u = 0; u < 4; ++u)
#pragma unroll
                        for (int c = 0; c < kPer; ++c) v[u][c] = __ldg(src0 + (j + u) * stride + c);
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const float wj = __shfl_sync(0xffffffffu, w, j + u);
#pragma unroll
                        for (int c = 0; c < kPer; ++c) acc[c] += wj * v[u][c];
                    }
                }
                for (; j < n; ++j) {
                    const float wj = __shfl_sync(0xffffffffu, w, j);
#pragma unroll
                    for (int c = 0; c < kPer; ++c) acc[c] += wj * __ldg(src0 + j * stride + c);
                }
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) lsum += __shfl_xor_sync(0xffffffffu, lsum, o);
        }
        const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
        uint16_t* dst = out + ((long)(q0 + r / g) * Hq + hk * g + r % g) * D + lane * kPer;
        if constexpr (kPer == 4)
            *reinterpret_cast<uint2*>(dst) = make_uint2(pack_bf16x2(acc[0] * inv, acc[1] * inv),
                                                        pack_bf16x2(acc[2] * inv, acc[3] * inv));
        else
            *reinterpret_cast<uint32_t*>(dst) = pack_bf16x2(acc[0] * inv, acc[1] * inv);
    }
}

// ------------------------------------------------------------ metadata -----
// One CTA: q_start (exclusive prefix sum of q_lens) and the list of query
// tiles (or tile pairs) of the sequences that take the tensor-core kernel,
// ordered by decreasing number of KV tiles (longest first) with a counting
// sort.  Entry = (sequence, first 128-row tile).
__global__ void __launch_bounds__(1024) paged_meta_kernel(const int32_t* __restrict__ ctx_lens,
                                                          const int32_t* __restrict__ q_lens, int num_seqs, int mbps,
                                                          int g, int causal, int tiles_per_entry,
                                                          int32_t* __restrict__ q_start, int32_t* __restrict__ count,
                                                          int32_t* __restrict__ list, int max_entries,
                                                          DevCtx ctx) {
    extern __shared__ int hist[];  // [nbins + 1]
    __shared__ int warp_sums[32];
    __shared__ int carry;
    const int nbins = (mbps * kBS + 127) / 128 + 1;
    for (int i = threadIdx.x; i <= nbins; i += blockDim.x) hist[i] = 0;
    if (threadIdx.x == 0) carry = 0;
    __syncthreads();
    // prefix sum of q_lens, 1024 sequences per pass
    for (int base = 0; base < num_seqs; base += blockDim.x) {
        const int s = base + threadIdx.x;
        int v = s < num_seqs ? q_lens[s] : 0;
        int x = v;
        const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        if (lane == 31) warp_sums[w] = x;
        __syncthreads();
        if (w == 0) {
            int t = warp_sums[lane];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                int y = __shfl_up_sync(0xffffffffu, t, o);
                if (lane >= o) t += y;
            }
            warp_sums[lane] = t;
        }
        __syncthreads();
        const int excl = carry + (w ? warp_sums[w - 1] : 0) + x - v;
        if (s < num_seqs) q_start[s] = excl;
        __syncthreads();
        if (threadIdx.x == blockDim.x - 1) carry = excl + v;
        __syncthreads();
    }
    if (threadIdx.x == 0) q_start[num_seqs] = carry;
    // histogram of entry costs
    auto entry_cost = [&](int ql, int cl, int t0) {
        const int last_row = min(ql, t0 + 128 * tiles_per_entry) - 1;  // last query row of the entry
        const int kv_end = causal ? cl - ql + last_row + 1 : cl;
        return (kv_end + 127) / 128;
    };
    for (int s = threadIdx.x; s < num_seqs; s += blockDim.x) {
        const int ql = q_lens[s], cl = ctx_lens[s];
        if (ql <= 0 || is_decode_row(ql, g)) continue;
        if (ql > cl || cl > mbps * kBS) {
            raise_error(ctx, ERR_BOUNDS_BIT);
            continue;
        }
        const int ntile = (ql + 127) / 128;
        for (int t = 0; t < ntile; t += tiles_per_entry) atomicAdd(&hist[entry_cost(ql, cl, t * 128)], 1);
    }
    __syncthreads();
    if (threadIdx.x == 0) {  // bucket starts, highest cost first
        int run = 0;
        for (int b = nbins - 1; b >= 0; --b) {
            const int c = hist[b];
            hist[b] = run;
            run += c;
        }
        hist[nbins] = run;
        *count = run < max_entries ? run : max_entries;
    }
    __syncthreads();
    for (int s = threadIdx.x; s < num_seqs; s += blockDim.x) {
        const int ql = q_lens[s], cl = ctx_lens[s];
        if (ql <= 0 || is_decode_row(ql, g) || ql > cl || cl > mbps * kBS) continue;
        const int ntile = (ql + 127) / 128;
        for (int t = 0; t < ntile; t += tiles_per_entry) {
            const int pos = atomicAdd(&hist[entry_cost(ql, cl, t * 128)], 1);
            if (pos < max_entries) {
                list[2 * pos] = s;
                list[2 * pos + 1] = t;
            }
        }
    }
}

template <int D>
static fa_status launch_decode(const void* q, const void* k_cache, const void* v_cache, const int32_t* bt,
                               const int32_t* ctx_lens, const int32_t* q_lens, void* out, const PagedWs& w,
                               uint8_t* ws, int num_seqs, int mbps, int num_blocks, int Hq, int Hkv, int causal,
                               float scale, cudaStream_t s, const DevCtx& ctx, int* launches) {
    CUtensorMap tk, tv;
    const uint64_t dims[4] = {(uint64_t)D, (uint64_t)kBS, (uint64_t)Hkv, (uint64_t)num_blocks};
    const uint64_t strides[3] = {(uint64_t)D * 2, (uint64_t)kBS * D * 2, (uint64_t)Hkv * kBS * D * 2};
    const uint32_t box[4] = {64, (uint32_t)kBS, 1, 1};
    fa_status st = encode_tmap_bf16_4d(&tk, k_cache, dims, strides, box);
    if (st != FA_OK) return st;
    if ((st = encode_tmap_bf16_4d(&tv, v_cache, dims, strides, box)) != FA_OK) return st;
    using L = DecodeSmem<D>;
    static bool attr_done = false;  // benign race: setting the attribute twice is harmless
    if (!attr_done) {
        if (cudaFuncSetAttribute(paged_decode_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kBytes) !=
            cudaSuccess)
            return FA_ERR_CUDA;
        attr_done = true;
    }
    float* part_o = reinterpret_cast<float*>(ws + w.part_o);
    float2* part_ml = reinterpret_cast<float2*>(ws + w.part_ml);
    const float scale_log2 = scale * 1.4426950408889634f;
    dim3 grid(w.max_splits, Hkv, num_seqs);
    paged_decode_kernel<D><<<grid, kDecodeWarps * 32, L::kBytes, s>>>(
        tk, tv, static_cast<const uint16_t*>(q), bt, ctx_lens, q_lens, static_cast<uint16_t*>(out), part_o,
        part_ml, mbps, num_blocks, Hq, Hkv, causal, scale_log2, w.split_blocks, w.max_splits, ctx);
    if (cudaGetLastError() != cudaSuccess) return FA_ERR_CUDA;
    ++*launches;
    if (w.max_splits > 1) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(num_seqs, Hkv);
        cfg.blockDim = dim3(kMergeThreads);
        cfg.stream = s;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (cudaLaunchKernelEx(&cfg, paged_merge_kernel<D>, ctx_lens, q_lens, static_cast<const float*>(part_o),
                               static_cast<const float2*>(part_ml), static_cast<uint16_t*>(out), Hq, Hkv,
                               w.split_blocks, w.max_splits, mbps) != cudaSuccess)
            return FA_ERR_CUDA;
        ++*launches;
    }
    return FA_OK;
}

}  // namespace fa

using namespace fa;

extern "C" {

size_t fa_paged_attn_workspace_size(int num_seqs, int max_blocks_per_seq, int Hq, int Hkv, int d, int total_q) {
    if (num_seqs < 0 || max_blocks_per_seq < 0 || Hq <= 0 || Hkv <= 0 || d <= 0 || total_q < 0) return 0;
    return paged_ws_layout(num_seqs, max_blocks_per_seq, Hq, Hkv, d, total_q).total;
}

fa_status fa_paged_attn(const void* q, const void* k_cache, const void* v_cache, const int32_t* block_table,
                        const int32_t* ctx_lens, const int32_t* q_lens, void* out, int num_seqs,
                        int max_blocks_per_seq, int num_blocks, int Hq, int Hkv, int d, int block_size, int causal,
                        float scale, int total_q, int max_q_len, void* ws, size_t ws_bytes, fa_stream_t stream) {
    set_launch_count(0);
    if (num_seqs < 0 || max_blocks_per_seq < 0 || num_blocks < 0 || Hq <= 0 || Hkv <= 0 || total_q < 0 ||
        max_q_len < 0 || !(scale > 0.f) || !(scale < INFINITY))
        return FA_ERR_INVALID_ARG;
    if (block_size != kBS || (d != 64 && d != 128) || Hq % Hkv != 0) return FA_ERR_UNSUPPORTED;
    if (num_seqs == 0 || total_q == 0 || max_q_len == 0) return FA_OK;
    if (!q || !k_cache || !v_cache || !block_table || !ctx_lens || !q_lens || !out) return FA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned32(out)) return FA_ERR_INVALID_ARG;
    if (num_blocks == 0 || max_blocks_per_seq == 0) return FA_ERR_INVALID_ARG;
    const PagedWs w = paged_ws_layout(num_seqs, max_blocks_per_seq, Hq, Hkv, d, total_q);
    if (!ws || ws_bytes < w.total || (reinterpret_cast<uintptr_t>(ws) & 255)) return FA_ERR_WORKSPACE;
    fa_status st = check_device();
    if (st != FA_OK) return st;
    DevCtx ctx;
    if ((st = make_ctx(&ctx)) != FA_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    uint8_t* wsb = static_cast<uint8_t*>(ws);
    const int g = Hq / Hkv;
    int launches = 0;
    if (g <= kDecodeRows) {
        st = d == 128 ? launch_decode<128>(q, k_cache, v_cache, block_table, ctx_lens, q_lens, out, w, wsb, num_seqs,
                                           max_blocks_per_seq, num_blocks, Hq, Hkv, causal, scale, s, ctx, &launches)
                      : launch_decode<64>(q, k_cache, v_cache, block_table, ctx_lens, q_lens, out, w, wsb, num_seqs,
                                          max_blocks_per_seq, num_blocks, Hq, Hkv, causal, scale, s, ctx, &launches);
        if (st != FA_OK) return st;
    }
    if (!is_decode_row(max_q_len, g)) {
        const int tiles_per_entry = (g % 2 == 0) ? 1 : 2;
        int32_t* q_start = reinterpret_cast<int32_t*>(wsb + w.q_start);
        int32_t* count = reinterpret_cast<int32_t*>(wsb + w.work_count);
        int32_t* list = reinterpret_cast<int32_t*>(wsb + w.work_list);
        const int nbins = (max_blocks_per_seq * kBS + 127) / 128 + 1;
        const size_t hist_bytes = sizeof(int) * (size_t)(nbins + 1);
        if (hist_bytes > 200 * 1024) return FA_ERR_UNSUPPORTED;
        if (hist_bytes > 48 * 1024 &&
            cudaFuncSetAttribute(paged_meta_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)hist_bytes) !=
                cudaSuccess)
            return FA_ERR_CUDA;
        paged_meta_kernel<<<1, 1024, hist_bytes, s>>>(ctx_lens, q_lens, num_seqs, max_blocks_per_seq, g, causal,
                                                      tiles_per_entry, q_start, count, list, w.max_entries, ctx);
        if (cudaGetLastError() != cudaSuccess) return FA_ERR_CUDA;
        ++launches;
        st = launch_paged_prefill(q, k_cache, v_cache, block_table, ctx_lens, q_lens, q_start, list, count, out,
                                  num_seqs, max_blocks_per_seq, num_blocks, Hq, Hkv, d, causal, scale, total_q, s,
                                  ctx);
        if (st != FA_OK) return st;
        ++launches;
    }
    set_launch_count(launches);
    return FA_OK;
}

}  // extern "C"

// ------------------------------------------------------ allocation-free ---
// Scratch for fa_paged_attn_noalloc: a fixed device array that every GPU
// loading this library holds until the process exits.  Host code only sees a
// stand-in for its name, so its device address is looked up per device with
// cudaGetSymbolAddress (with that device current) and handed to the kernels.
namespace fa {
namespace {
static __device__ __align__(256) uint8_t g_noalloc_scratch[FA_NOALLOC_SCRATCH_BYTES];
std::mutex g_noalloc_mu;
void* g_noalloc_ptr[64] = {};

fa_status noalloc_scratch(void** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return FA_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return FA_ERR_CUDA;
        g_noalloc_ptr[dev] = p;
    }
    *out = g_noalloc_ptr[dev];
    return FA_OK;
}
}  // namespace
}  // namespace fa

extern "C" fa_status fa_paged_attn_noalloc(const void* q, const void* k_cache, const void* v_cache,
                                           const int32_t* block_table, const int32_t* ctx_lens,
                                           const int32_t* q_lens, void* out, int num_seqs, int max_blocks_per_seq,
                                           int num_blocks, int Hq, int Hkv, int d, int block_size, int causal,
                                           float scale, int total_q, int max_q_len, fa_stream_t stream) {
    const size_t need = fa_paged_attn_workspace_size(num_seqs, max_blocks_per_seq, Hq, Hkv, d, total_q);
    if (need > FA_NOALLOC_SCRATCH_BYTES) return FA_ERR_WORKSPACE;  // problem too large for the fixed scratch
    void* scratch = nullptr;
    fa_status st = fa::noalloc_scratch(&scratch);
    if (st != FA_OK) return st;
    return fa_paged_attn(q, k_cache, v_cache, block_table, ctx_lens, q_lens, out, num_seqs, max_blocks_per_seq,
                         num_blocks, Hq, Hkv, d, block_size, causal, scale, total_q, max_q_len, scratch,
                         FA_NOALLOC_SCRATCH_BYTES, stream);
}
