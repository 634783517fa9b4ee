// Paged attention ("Fast Attention Kernels and Operator Fusion", section
// "Paged Attention Kernels"): keys and values sit in 16-token blocks of a
// shared pool, [num_blocks, Hkv, 16, d] bf16, and every access goes through
// the per-sequence block table ("the kernel cannot assume that K[t+1] is
// adjacent to K[t]").
//
// Decode rows (the section "FlashAttention-Style Kernels" notes that decode
// has one or a few queries and is dominated by reading the growing cache)
// take a bandwidth-bound kernel that streams the cache in balanced ranges:
//   * the (sequence, kv head) segments are laid end to end as one stream of
//     16-token pages; each of the grid's warps (one CTA of eight warps per SM)
//     takes an equal contiguous range of pages, so every SM moves the same
//     number of bytes whatever the mix of context lengths;
//   * each warp streams its pages through a private ring of shared memory
//     with TMA (one 2 KB box per 64 channels of K and of V, 128-byte swizzled
//     so the fragment loads below are bank-conflict free); the physical block
//     id is read from the block table just before the copy;
//   * all Hq/Hkv query heads of the kv head (times the chunk's query tokens,
//     at most 16 rows) share each K/V load: they form the M dimension of
//     m16n8k16 warp MMAs, so K and V are read from HBM exactly once;
//   * the running row max / row sum are kept in fp32 (online softmax with
//     base-2 exponentials, scale * log2(e) folded into the scores);
//   * a segment inside one warp's range is written as final bf16 output; a
//     segment cut by a range boundary leaves fp32 partials (unnormalised O,
//     running max, running sum) in shared memory, which the CTA combines with
//     log-sum-exp weights once its warps are done: into the final rows when
//     the segment lies inside the CTA's range, otherwise into one partial per
//     CTA that a second kernel merges the same way.
// Longer chunks take the tensor-core kernel (attn_tc.cu) through a work list
// built on the device by `paged_meta_kernel`.
#include <algorithm>
#include <mutex>
#include <type_traits>

#include "host_common.cuh"

namespace fa {

constexpr int kBS = 16;            // tokens per block
constexpr int kDecodeRows = 16;    // M of the warp MMA

// Launched from attn_tc.cu.
fa_status launch_paged_prefill(const void* q, const void* k_cache, const void* v_cache, const int32_t* block_table,
                               const int32_t* ctx_lens, const int32_t* q_lens, const int32_t* q_start,
                               const int32_t* work_list, const int32_t* work_count, void* out, int num_seqs,
                               int mbps, int num_blocks, int Hq, int Hkv, int d, int causal, float scale,
                               int total_q, cudaStream_t s, const DevCtx& ctx);

__host__ __device__ inline bool is_decode_row(int q_len, int g) { return q_len >= 1 && g * q_len <= kDecodeRows; }

// ------------------------------------------------------------------ layout --
constexpr int kStreamWarps = 8;      // page streams per decode CTA
constexpr int kMaxStreamCtas = 160;  // decode grid cap (one CTA per SM); sizes the partial slots

struct PagedWs {
    size_t q_start, work_count, work_list, part_o, part_ml, total;
    int max_entries;
};

// Workspace: scheduling lists of the tensor-core path, then two partial slots
// per decode CTA (16 rows of fp32 O, plus (max, sum) per row).
inline PagedWs paged_ws_layout(int num_seqs, int mbps, int Hq, int Hkv, int d, int total_q) {
    (void)Hq;
    (void)Hkv;
    (void)mbps;
    PagedWs w{};
    w.max_entries = total_q / 16 + num_seqs + 1;  // entries hold at least 16 tokens (paged_tc_entry_tokens)
    size_t off = 0;
    w.q_start = off;
    off = align256(off + sizeof(int32_t) * (size_t)(num_seqs + 1));
    w.work_count = off;
    off = align256(off + sizeof(int32_t) * 4);
    w.work_list = off;
    off = align256(off + sizeof(int32_t) * 2 * (size_t)w.max_entries);
    w.part_o = off;
    off = align256(off + sizeof(float) * (size_t)2 * kMaxStreamCtas * kDecodeRows * d);
    w.part_ml = off;
    off = align256(off + sizeof(float2) * (size_t)2 * kMaxStreamCtas * kDecodeRows);
    w.total = off;
    return w;
}

// -------------------------------------------------------------- decode -----
// Work is balanced by pages: the decode segments (sequence, kv head) are laid
// end to end, sequence-major, as one stream of 16-token pages; warp w of the
// grid takes pages [w*P/W, (w+1)*P/W), so CTA c holds pages [8c*P/W,
// (8c+8)*P/W).  A segment that lies inside one warp's range is finished by
// that warp (bf16 output); a segment cut by a warp's range boundary leaves
// that warp's partial (running max, row sum, unnormalised O) in shared memory,
// and the CTA combines the pieces of its warps: final rows for a segment inside
// the CTA's range, else the CTA's partial in slot 2c (the CTA's first segment)
// or 2c+1 (its last) for the merge kernel.  Every page is read once; every warp
// streams the same number of bytes, so no SM waits on a long sequence.

// Pages one kv head of sequence s contributes to the decode stream (0 when the
// sequence takes the tensor-core path or its lengths are inconsistent).
__device__ __forceinline__ int decode_blocks(const int32_t* __restrict__ q_lens, const int32_t* __restrict__ ctx_lens,
                                             int s, int g, int mbps) {
    const int ql = __ldg(q_lens + s), cl = __ldg(ctx_lens + s);
    if (!is_decode_row(ql, g) || ql > cl || cl > mbps * kBS) return 0;
    return (cl + kBS - 1) / kBS;
}

// The stream partition: warp w of W starts at page floor(w * P / W).  With
// P = qt * W + rm this is w * qt + (w * rm) / W, where (w * rm) < W * W fits
// 32 bits: one 64-bit division per kernel instead of one per lookup.
struct StreamSplit {
    long long P, qt;
    int rm, W;
    __device__ StreamSplit(long long P_, int W_) : P(P_), qt(P_ / W_), rm((int)(P_ - P_ / W_ * W_)), W(W_) {}
    __device__ __forceinline__ long long begin(int w) const {
        return (long long)w * qt + (int)((unsigned)w * (unsigned)rm / (unsigned)W);
    }
    // warp whose range holds page x (0 <= x < P)
    __device__ __forceinline__ int owner(long long x) const {
        int w = (int)min((long long)W - 1, x * W / P);  // within one of the owner
        while (w + 1 < W && begin(w + 1) <= x) ++w;
        while (w > 0 && begin(w) > x) --w;
        return w;
    }
};

// Shared memory of a decode CTA: each warp's TMA ring, then each warp's slot
// for the partial of its first segment (ROWS query rows).  The ring has three
// stages (8 KB each at d = 128, 4 KB at d = 64) except at d = 128 with slots of
// 16 rows, which leave room for two; the 8-bit (E4M3) cache's pages are half
// the bytes, so its ring is twice as deep to keep the same bytes in flight.
template <int D, bool KV8, int ROWS>
struct StreamSmem {
    static constexpr int kPage = kBS * D * (KV8 ? 1 : 2);  // bytes of one K (or V) page
    static constexpr int kStage = 2 * kPage;              // K page + V page
    static constexpr int kStages = (KV8 ? 2 : 1) * (D == 128 && ROWS > 6 ? 2 : 3);
    static constexpr int kRing = kStreamWarps * kStages * kStage;
    // a partial: ROWS rows of unnormalised O (fp32, rows kSlotRow floats
    // apart), then (max, sum) per row
    static constexpr int kSlotRow = D + 8;
    static constexpr int kSlotBytes = ROWS * kSlotRow * 4 + ROWS * 8;
    static constexpr int kSlots = kStreamWarps * kSlotBytes;
    static constexpr int kBars = kStreamWarps * kStages + 1;
    static constexpr int kCutEntries = 2 * kStreamWarps;  // segments cut between the CTA's warps, at most
    static constexpr int kBytes = 1024 /*align slack*/ + kRing + kSlots + kBars * 8 + 64 + kCutEntries * 32;
    static_assert(kSlotBytes <= kStages * kStage, "a warp's ring holds the partial of its last segment");
    static_assert(kSlots % 64 == 0 && kSlotBytes % 16 == 0, "slots keep 16-byte alignment");
    static_assert((kStreamWarps * kStages * 8) % 64 == 0, "the barrier after the ring barriers is 64-byte aligned");
};

// Position of a stream cursor: sequence, kv head, block within the sequence.
struct Cursor {
    int s, hk, blk, nblk;  // nblk: pages per kv head of sequence s
    int q0;                // first packed query row of sequence s
};

// KV8 reads the 8-bit cache: K pages [16 tokens][D] bytes (128-byte swizzled
// rows), V pages [D channels][16 tokens] bytes; the warp MMAs run in f16
// (every E4M3 value is an f16 value; bf16 queries are converted to f16),
// k_scale is folded into scale_log2 by the host and v_scale multiplies the
// output.  The MMA's K dimension is taken in a permuted order so that one
// ldmatrix lane word (4 consecutive bytes = 4 channels, or 4 tokens of V)
// gives both B registers: logical k (2t, 2t+1, 2t+8, 2t+9) of a 16-wide step
// = elements (4t .. 4t+3); queries are loaded in the same order for Q K^T,
// and for P V the S tile's columns (tokens) are produced in that order by
// loading K rows 4t+2nt+e into n-tile nt, column 2t+e.
constexpr int kLensPerLane = 8;  // sequences per lane whose lengths are loaded in one batch
template <int D, bool KV8, int ROWS>
__global__ void __launch_bounds__(kStreamWarps * 32, 1)
    paged_decode_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                        const uint16_t* __restrict__ q, const int32_t* __restrict__ bt,
                        const int32_t* __restrict__ ctx_lens, const int32_t* __restrict__ q_lens,
                        uint16_t* __restrict__ out, float* __restrict__ part_o, float2* __restrict__ part_ml,
                        int num_seqs, int mbps, int num_blocks, int Hq, int Hkv, int q_prefetch_rows, int causal,
                        float scale_log2, float v_scale, DevCtx ctx) {
    // the merge kernel that follows may be scheduled now; it waits for this
    // grid's completion before reading anything
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    using L = StreamSmem<D, KV8, ROWS>;
    constexpr int kStreamStages = L::kStages;  // ring depth of this variant
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kRing + L::kSlots);
    uint64_t* never = bars + kStreamWarps * kStreamStages;  // nothing arrives on it (time-out test hook)
    volatile int* abort_flag = reinterpret_cast<volatile int*>(never + 1);
    int* cut_count = const_cast<int*>(abort_flag) + 1;  // entries in cut_table
    // 2 int4 per entry, see the end; `never` is 64-byte aligned (the ring, the
    // slots and the barriers before it are multiples of 64 bytes), so this is 16
    int4* cut_table = reinterpret_cast<int4*>(never + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = Hq / Hkv;
    const int W = gridDim.x * kStreamWarps;
    const int gw = blockIdx.x * kStreamWarps + warp;
    if (threadIdx.x == 0) {
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
        for (int i = 0; i < L::kBars; ++i) mbar_init(&bars[i], 1);
        *abort_flag = 0;
        *cut_count = 0;
        mbar_fence_init();
    }
    {
        // warm L2 with this CTA's share of the block table and (when every
        // query row is a decode row) of the queries, read right after the lengths
        constexpr long kMaxPrefetchLines = (4L << 20) / 128;  // 4 MB each at most
        const long tb_lines = min(kMaxPrefetchLines, ((long)num_seqs * mbps * 4 + 127) / 128);
        const long q_lines = min(kMaxPrefetchLines, ((long)q_prefetch_rows * Hq * D * 2 + 127) / 128);
        const long tb_lo = tb_lines * blockIdx.x / gridDim.x, tb_hi = tb_lines * (blockIdx.x + 1) / gridDim.x;
        const long q_lo = q_lines * blockIdx.x / gridDim.x, q_hi = q_lines * (blockIdx.x + 1) / gridDim.x;
        for (long i = tb_lo + threadIdx.x; i < tb_hi; i += blockDim.x)
            asm volatile("prefetch.global.L2 [%0];" ::"l"(reinterpret_cast<const char*>(bt) + i * 128));
        for (long i = q_lo + threadIdx.x; i < q_hi; i += blockDim.x)
            asm volatile("prefetch.global.L2 [%0];" ::"l"(reinterpret_cast<const char*>(q) + i * 128));
    }

    // Where this warp's pages start.  Every warp finds out on its own (no
    // CTA-wide step on the path to the first copy): lane j sums the decode
    // pages and the query rows of sequences [j*per, (j+1)*per), and a warp
    // scan gives each lane's offsets and the total P.
    const int per = (num_seqs + 31) >> 5;
    const int s_lo = min(num_seqs, lane * per), s_hi = min(num_seqs, s_lo + per);
    long long my_p = 0, my_q = 0;
    bool bad = false;
    auto count = [&](int ql, int cl) {
        my_q += ql;
        if (!is_decode_row(ql, g)) return;
        if (ql > cl || cl > mbps * kBS) {
            bad = true;
            return;
        }
        my_p += (long long)Hkv * ((cl + kBS - 1) / kBS);
    };
    if (per <= kLensPerLane) {
        int qv[kLensPerLane], cv[kLensPerLane];
#pragma unroll
        for (int i = 0; i < kLensPerLane; ++i) {  // all loads issued before any is used
            const bool in = s_lo + i < s_hi;
            qv[i] = in ? __ldg(q_lens + s_lo + i) : 0;
            cv[i] = in ? __ldg(ctx_lens + s_lo + i) : 0;
        }
        __syncthreads();  // barrier initialisation visible to every warp (the loads are in flight)
#pragma unroll
        for (int i = 0; i < kLensPerLane; ++i)
            if (s_lo + i < s_hi) count(qv[i], cv[i]);
    } else {
        __syncthreads();
#pragma unroll 4
        for (int s = s_lo; s < s_hi; ++s) count(__ldg(q_lens + s), __ldg(ctx_lens + s));
    }
    if (bad && gw == 0) raise_error(ctx, ERR_BOUNDS_BIT);
    long long inc_p = my_p, inc_q = my_q;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const long long yp = __shfl_up_sync(0xffffffffu, inc_p, o), yq = __shfl_up_sync(0xffffffffu, inc_q, o);
        if (lane >= o) {
            inc_p += yp;
            inc_q += yq;
        }
    }
    const long long P = __shfl_sync(0xffffffffu, inc_p, 31);
    if (P == 0) return;
    const StreamSplit split(P, W);
    const long long b0 = split.begin(gw), b1 = split.begin(gw + 1);
    const int n_pages = (int)(b1 - b0);
    if (n_pages <= 0) return;  // not among the warps of the CTA barrier at the end
    // the lane whose sequences hold page b0 walks them (lengths are L1 hits now)
    Cursor start;
    {
        const unsigned hit = __ballot_sync(0xffffffffu, my_p > 0 && b0 >= inc_p - my_p && b0 < inc_p);
        const int src = __ffs(hit) - 1;  // exactly one lane: 0 <= b0 < P
        int a_s = 0, a_off = 0, a_q0 = 0;
        if (lane == src) {
            long long off = b0 - (inc_p - my_p), q0 = inc_q - my_q;
            for (int s = s_lo; s < s_hi; ++s) {
                const int ql = __ldg(q_lens + s), cl = __ldg(ctx_lens + s);
                const long long n =
                    (is_decode_row(ql, g) && ql <= cl && cl <= mbps * kBS) ? (long long)Hkv * ((cl + kBS - 1) / kBS)
                                                                            : 0;
                if (off < n) {
                    a_s = s;
                    a_off = (int)off;
                    a_q0 = (int)q0;
                    break;
                }
                off -= n;
                q0 += ql;
            }
        }
        start.s = __shfl_sync(0xffffffffu, a_s, src);
        a_off = __shfl_sync(0xffffffffu, a_off, src);
        start.q0 = __shfl_sync(0xffffffffu, a_q0, src);
        start.nblk = decode_blocks(q_lens, ctx_lens, start.s, g, mbps);
        start.hk = a_off / start.nblk;
        start.blk = a_off % start.nblk;
    }

    uint8_t* ring = smem + warp * kStreamStages * L::kStage;
    uint64_t* wbar = bars + warp * kStreamStages;
    // Partials of segments cut by a range boundary stay in shared memory:
    // the first segment's in this warp's slot, the last one's (when it is
    // another segment) in this warp's ring, free once its last page is read.
    float* slot_first = reinterpret_cast<float*>(smem + L::kRing + warp * L::kSlotBytes);
    float* slot_last = reinterpret_cast<float*>(ring);
    // advances a cursor by one page; entering a new sequence skips the ones
    // with no decode pages and carries the packed query offset along
    auto advance = [&](Cursor& c) {
        if (++c.blk < c.nblk) return;
        c.blk = 0;
        if (++c.hk < Hkv) return;
        c.hk = 0;
        do {
            c.q0 += __ldg(q_lens + c.s);
            ++c.s;
            c.nblk = c.s < num_seqs ? decode_blocks(q_lens, ctx_lens, c.s, g, mbps) : 0;
        } while (c.s < num_seqs && c.nblk == 0);
    };

    Cursor ci = start;  // issue cursor (lane 0 only)
    // lane 0 reads the block-table entry of the next page one issue ahead, so
    // that load's latency is not on the copy's path
    int next_phys = lane == 0 ? __ldg(bt + (long)ci.s * mbps + ci.blk) : 0;
    auto issue = [&](int i) {
        const int stage = i % kStreamStages;
        int phys = next_phys;
        if (phys < 0 || phys >= num_blocks) {
            raise_error(ctx, ERR_BOUNDS_BIT);
            phys = num_blocks;  // outside the tensor map: the copy fills zeros
        }
        uint8_t* kp = ring + stage * L::kStage;
        uint8_t* vp = kp + L::kPage;
        mbar_arrive_expect_tx(&wbar[stage], L::kStage);
        if constexpr (KV8) {  // one box per page: K rows, V channel rows
            tma_load_4d(kp, &tm_k, &wbar[stage], 0, 0, ci.hk, phys);
            tma_load_4d(vp, &tm_v, &wbar[stage], 0, 0, ci.hk, phys);
        } else {
#pragma unroll
            for (int h = 0; h < D / 64; ++h) {
                tma_load_4d(kp + h * 2048, &tm_k, &wbar[stage], h * 64, 0, ci.hk, phys);
                tma_load_4d(vp + h * 2048, &tm_v, &wbar[stage], h * 64, 0, ci.hk, phys);
            }
        }
        advance(ci);
        if (i + 1 < n_pages) next_phys = __ldg(bt + (long)ci.s * mbps + ci.blk);
    };
    bool ok = !ctx.force_timeout || mbar_wait_warp(never, 0, ctx.wait_ns, abort_flag);
    if (!ok && lane == 0) {
        raise_error(ctx, ERR_TIMEOUT_BIT);
        *abort_flag = 1;
    }
    int issued = 0;  // lane 0's count of copies issued
    if (lane == 0 && ok)
        for (; issued < n_pages && issued < kStreamStages; ++issued) issue(issued);

    const int gid = lane >> 2, tig = lane & 3, mi = lane >> 3, r8 = lane & 7;
    Cursor cc = start;            // compute cursor (all lanes)
    long long seg_first = b0 - start.blk;  // global index of the current segment's first page
    Cursor seg_last = start;               // the segment begun last, its first page and query rows
    long long seg_last_first = seg_first;
    int seg_last_rows = 0, first_rows = -1;  // and the first segment's query rows
    int ctx_len = 0, q_len = 0, nrows = 0, pos_r0 = 0, pos_r1 = 0;
    uint32_t qa[D / 16][4];
    float o[D / 8][4];
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;

    // starts segment (cc.s, cc.hk): loads its query rows as MMA A fragments
    // (rows r = token * g + head-in-group) and resets the softmax state
    auto begin_segment = [&]() {
        seg_last = cc;
        seg_last_first = seg_first;
        ctx_len = __ldg(ctx_lens + cc.s);
        q_len = __ldg(q_lens + cc.s);
        nrows = g * q_len;
        seg_last_rows = nrows;
        if (first_rows < 0) first_rows = nrows;
        const int rr[2] = {gid, gid + 8};
        const uint16_t* qrow[2];
#pragma unroll
        for (int i = 0; i < 2; ++i)
            qrow[i] = rr[i] < nrows ? q + ((long)(cc.q0 + rr[i] / g) * Hq + cc.hk * g + rr[i] % g) * D : nullptr;
        if constexpr (KV8) {
            // f16, channels 4t .. 4t+3 of each 16-channel step (the permuted K order)
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks) {
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    const uint2 w = qrow[i] ? __ldg(reinterpret_cast<const uint2*>(qrow[i] + ks * 16 + tig * 4))
                                            : make_uint2(0u, 0u);
                    qa[ks][i] = pack_f16x2(__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xFFFF0000u));
                    qa[ks][i + 2] = pack_f16x2(__uint_as_float(w.y << 16), __uint_as_float(w.y & 0xFFFF0000u));
                }
            }
        } else {
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks) {
                const int c = ks * 16 + tig * 2;
                qa[ks][0] = qrow[0] ? __ldg(reinterpret_cast<const uint32_t*>(qrow[0] + c)) : 0u;
                qa[ks][1] = qrow[1] ? __ldg(reinterpret_cast<const uint32_t*>(qrow[1] + c)) : 0u;
                qa[ks][2] = qrow[0] ? __ldg(reinterpret_cast<const uint32_t*>(qrow[0] + c + 8)) : 0u;
                qa[ks][3] = qrow[1] ? __ldg(reinterpret_cast<const uint32_t*>(qrow[1] + c + 8)) : 0u;
            }
        }
        // keys <= pos(row) are visible
        pos_r0 = causal ? ctx_len - q_len + gid / g : ctx_len - 1;
        pos_r1 = causal ? ctx_len - q_len + (gid + 8) / g : ctx_len - 1;
#pragma unroll
        for (int n = 0; n < D / 8; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
        m0 = m1 = -INFINITY;
        l0 = l1 = 0.f;
    };
    // finishes the current segment: final bf16 rows when the whole segment
    // was in this warp's range, otherwise a partial in shared memory
    auto end_segment = [&]() {
        float la = l0 + __shfl_xor_sync(0xffffffffu, l0, 1);
        la += __shfl_xor_sync(0xffffffffu, la, 2);
        float lb = l1 + __shfl_xor_sync(0xffffffffu, l1, 1);
        lb += __shfl_xor_sync(0xffffffffu, lb, 2);
        const bool whole = seg_first >= b0 && seg_first + cc.nblk <= b1;
        const int rr[2] = {gid, gid + 8};
        const float ml[2] = {m0, m1}, ls[2] = {la, lb};
        if (whole) {
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const int r = rr[i];
                if (r >= nrows) continue;
                const float inv = ls[i] > 0.f ? v_scale / ls[i] : 0.f;
                uint16_t* dst = out + ((long)(cc.q0 + r / g) * Hq + cc.hk * g + r % g) * D;
#pragma unroll
                for (int n = 0; n < D / 8; ++n)
                    *reinterpret_cast<uint32_t*>(dst + n * 8 + tig * 2) =
                        pack_bf16x2(o[n][2 * i] * inv, o[n][2 * i + 1] * inv);
            }
        } else {
            // a slot holds ROWS rows: more means max_q_len was below a chunk's length
            if (nrows > ROWS && lane == 0) raise_error(ctx, ERR_BOUNDS_BIT);
            float* so = seg_first <= b0 ? slot_first : slot_last;
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const int r = rr[i];
                if (r >= nrows || r >= ROWS) continue;
#pragma unroll
                for (int n = 0; n < D / 8; ++n)
                    *reinterpret_cast<float2*>(so + r * L::kSlotRow + n * 8 + tig * 2) =
                        make_float2(o[n][2 * i] * v_scale, o[n][2 * i + 1] * v_scale);
                if (tig == 0) reinterpret_cast<float2*>(so + ROWS * L::kSlotRow)[r] = make_float2(ml[i], ls[i]);
            }
        }
    };

    int consumed = 0;
    if (ok) begin_segment();
    for (int i = 0; ok && i < n_pages; ++i, consumed = i) {
        if (i > 0 && cc.blk == 0) {  // the cursor entered a new segment
            seg_first = b0 + i;
            begin_segment();
        }
        const int stage = i % kStreamStages;
        if (!mbar_wait_warp(&wbar[stage], (i / kStreamStages) & 1, ctx.wait_ns, abort_flag)) {
            if (lane == 0) {
                raise_error(ctx, ERR_TIMEOUT_BIT);
                *abort_flag = 1;
            }
            ok = false;
            break;
        }
        const uint32_t kbase = smem_u32(ring + stage * L::kStage);
        const uint32_t vbase = kbase + L::kPage;
        const int tok0 = cc.blk * kBS;

        // S = Q K^T : 16 rows x 16 tokens
        float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
        if constexpr (KV8) {
            // matrix mi: n-tile mi & 1, 16-byte chunk 2j + (mi >> 1); its row r8
            // is token 4 (r8 / 2) + 2 (mi & 1) + r8 % 2 (the S column order P V uses)
            const int tok = (r8 >> 1) * 4 + 2 * (mi & 1) + (r8 & 1);
#pragma unroll
            for (int j = 0; j < D / 32; ++j) {
                const int chunk = 2 * j + (mi >> 1);
                uint32_t w[4], b[8];
                ldsm_x4(kbase + tok * D + ((chunk ^ (tok & 7)) << 4), w[0], w[1], w[2], w[3]);
#pragma unroll
                for (int m = 0; m < 4; ++m) e4m3x4_to_f16x4(w[m], b[2 * m], b[2 * m + 1]);
                mma_f16_16816(sc[0], qa[2 * j], b[0], b[1]);
                mma_f16_16816(sc[1], qa[2 * j], b[2], b[3]);
                mma_f16_16816(sc[0], qa[2 * j + 1], b[4], b[5]);
                mma_f16_16816(sc[1], qa[2 * j + 1], b[6], b[7]);
            }
        } else {
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks) {
                const int tok = (mi >> 1) * 8 + r8;
                const int chunk = ks * 2 + (mi & 1);
                uint32_t b0r, b1r, b2r, b3r;
                ldsm_x4(kbase + (chunk >> 3) * 2048 + sw128_offset(tok, chunk & 7), b0r, b1r, b2r, b3r);
                mma_bf16_16816(sc[0], qa[ks], b0r, b1r);
                mma_bf16_16816(sc[1], qa[ks], b2r, b3r);
            }
        }
        // mask + online softmax (base 2)
        float x[2][4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int t = KV8 ? tok0 + tig * 4 + nt * 2 + (e & 1) : tok0 + nt * 8 + tig * 2 + (e & 1);
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
        float pr[2][4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            pr[nt][0] = fast_exp2(x[nt][0] - mu0);
            pr[nt][1] = fast_exp2(x[nt][1] - mu0);
            pr[nt][2] = fast_exp2(x[nt][2] - mu1);
            pr[nt][3] = fast_exp2(x[nt][3] - mu1);
        }
        l0 = l0 * a0 + (pr[0][0] + pr[0][1] + pr[1][0] + pr[1][1]);
        l1 = l1 * a1 + (pr[0][2] + pr[0][3] + pr[1][2] + pr[1][3]);
        if (__any_sync(0xffffffffu, a0 != 1.f || a1 != 1.f)) {
#pragma unroll
            for (int n = 0; n < D / 8; ++n) {
                o[n][0] *= a0;
                o[n][1] *= a0;
                o[n][2] *= a1;
                o[n][3] *= a1;
            }
        }
        uint32_t pa[4];
        if constexpr (KV8) {
            pa[0] = pack_f16x2(pr[0][0], pr[0][1]);
            pa[1] = pack_f16x2(pr[0][2], pr[0][3]);
            pa[2] = pack_f16x2(pr[1][0], pr[1][1]);
            pa[3] = pack_f16x2(pr[1][2], pr[1][3]);
        } else {
            pa[0] = pack_bf16x2(pr[0][0], pr[0][1]);
            pa[1] = pack_bf16x2(pr[0][2], pr[0][3]);
            pa[2] = pack_bf16x2(pr[1][0], pr[1][1]);
            pa[3] = pack_bf16x2(pr[1][2], pr[1][3]);
        }
        // O += P V : V rows past the context are zeroed so stale cache words
        // (possibly NaN) cannot reach the accumulator through a zero weight
        const int nvalid = ctx_len - tok0;  // >= 1
        if constexpr (KV8) {
            // V page rows are channels (16 token bytes each); matrix mi of
            // step q4 is n-tile 4 q4 + mi; a lane word holds tokens 4t .. 4t+3
            const uint32_t zb = (tig * 4 < nvalid ? 0x000000ffu : 0u) | (tig * 4 + 1 < nvalid ? 0x0000ff00u : 0u) |
                                (tig * 4 + 2 < nvalid ? 0x00ff0000u : 0u) | (tig * 4 + 3 < nvalid ? 0xff000000u : 0u);
#pragma unroll
            for (int q4 = 0; q4 < D / 32; ++q4) {
                uint32_t w[4];
                ldsm_x4(vbase + ((4 * q4 + mi) * 8 + r8) * 16, w[0], w[1], w[2], w[3]);
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    uint32_t b0r, b1r;
                    e4m3x4_to_f16x4(w[m] & zb, b0r, b1r);
                    mma_f16_16816(o[4 * q4 + m], pa, b0r, b1r);
                }
            }
        } else {
            const uint32_t zlo =
                (tig * 2 < nvalid ? 0x0000ffffu : 0u) | (tig * 2 + 1 < nvalid ? 0xffff0000u : 0u);
            const uint32_t zhi =
                (tig * 2 + 8 < nvalid ? 0x0000ffffu : 0u) | (tig * 2 + 9 < nvalid ? 0xffff0000u : 0u);
#pragma unroll
            for (int dn = 0; dn < D / 16; ++dn) {
                const int tok = (mi & 1) * 8 + r8;
                const int chunk = dn * 2 + (mi >> 1);
                uint32_t b0r, b1r, b2r, b3r;
                ldsm_x4_t(vbase + (chunk >> 3) * 2048 + sw128_offset(tok, chunk & 7), b0r, b1r, b2r, b3r);
                b0r &= zlo;
                b2r &= zlo;
                b1r &= zhi;
                b3r &= zhi;
                mma_bf16_16816(o[2 * dn], pa, b0r, b1r);
                mma_bf16_16816(o[2 * dn + 1], pa, b2r, b3r);
            }
        }
        __syncwarp();
        if (lane == 0 && issued < n_pages) issue(issued++);
        // leaving the segment: last page of the range or of the segment
        const bool last_here = (i + 1 == n_pages) || (cc.blk + 1 == cc.nblk);
        if (last_here) end_segment();
        advance(cc);
    }
    if (!ok && lane == 0) {
        // drain: let the copies this warp issued but did not consume land
        // before the CTA can exit
        for (int i = consumed; i < issued; ++i)
            (void)mbar_wait_bounded(&wbar[i % kStreamStages], (i / kStreamStages) & 1, 1000000000ull, nullptr);
    }

    // Segments cut between this CTA's warps (or by the CTA's range boundaries).
    // The warp holding a segment's first page within the CTA's range lists it;
    // then the CTA's warps share out the listed rows and combine the pieces of
    // the CTA's warps, from shared memory, with log-sum-exp weights: into the
    // final bf16 rows when the segment lies inside the CTA's range, otherwise
    // into the CTA's partial (slot 2c for the segment holding the CTA's first
    // page, 2c+1 for the one holding its last) for the merge kernel.  Warps
    // without pages have left; the barriers count the others.
    const int cw0 = blockIdx.x * kStreamWarps;
    long long wb[kStreamWarps + 1];  // first page of each warp of this CTA, then the CTA's end
#pragma unroll
    for (int w = 0; w <= kStreamWarps; ++w) wb[w] = split.begin(cw0 + w);
    unsigned busy = 0;  // warps of this CTA with pages
#pragma unroll
    for (int w = 0; w < kStreamWarps; ++w) busy |= (wb[w + 1] > wb[w] ? 1u : 0u) << w;
    const int nbusy = __popc(busy);
    asm volatile("bar.sync 1, %0;" ::"r"(32 * nbusy) : "memory");
    if (*abort_flag) return;
    const long long c0 = wb[0], c1 = wb[kStreamWarps];
    // 1. the warp holding a cut segment's first page within the CTA lists it:
    //    (first query row, kv head, rows, pieces) and (output kind, slot, source slot of its own piece)
    for (int which = 0; which < 2; ++which) {
        const Cursor X = which ? seg_last : start;
        const long long sf = which ? seg_last_first : b0 - start.blk;
        if (which == 1 && sf == b0 - start.blk) break;  // one segment only
        const long long se = sf + X.nblk;
        if (sf >= b0 && se <= b1) continue;  // finished by this warp
        if (sf < b0 && b0 > c0) continue;    // an earlier warp of the CTA holds its first piece here
        // pieces: this warp and the later warps of the CTA whose pages start
        // before the segment's end (warps without pages wrote nothing)
        const long long lim = min(se, c1);
        unsigned mask = 0;
#pragma unroll
        for (int w = 0; w < kStreamWarps; ++w)
            if (w >= warp && wb[w] < lim && ((busy >> w) & 1u)) mask |= 1u << w;
        if (lane == 0) {
            const int e = atomicAdd(cut_count, 1);  // < kCutEntries: at most two per warp
            const bool final_rows = sf >= c0 && se <= c1;
            cut_table[2 * e] = make_int4(X.q0, X.hk, min(ROWS, which ? seg_last_rows : first_rows), (int)mask);
            cut_table[2 * e + 1] = make_int4(final_rows ? -1 : 2 * (int)blockIdx.x + (sf <= c0 ? 0 : 1), warp, which, 0);
        }
    }
    asm volatile("bar.sync 1, %0;" ::"r"(32 * nbusy) : "memory");
    // 2. the CTA's warps share out the listed segments' rows: per row, the
    //    pieces are combined with log-sum-exp weights into the final bf16 row
    //    (segment inside the CTA's range) or the CTA's partial for the merge kernel
    const int n_cut = *cut_count;
    const int rank = __popc(busy & ((1u << warp) - 1u));
    constexpr int kPer = D / 32;  // channels per lane
    int e = 0, e_row0 = 0;        // entry of the current item, and its first item index
    for (int it = rank;; it += nbusy) {
        int4 h = make_int4(0, 0, 0, 0);
        while (e < n_cut) {
            h = cut_table[2 * e];
            if (it < e_row0 + h.z) break;
            e_row0 += h.z;
            ++e;
        }
        if (e >= n_cut) break;
        const int4 t = cut_table[2 * e + 1];
        const int r = it - e_row0;
        const unsigned mask = (unsigned)h.w;
        // piece of warp w: the listing warp's own slot (first or last segment), else warp w's first-segment slot
        auto piece = [&](int w) -> const float* {
            if (w == t.y && t.z) return reinterpret_cast<const float*>(smem + w * kStreamStages * L::kStage);
            return reinterpret_cast<const float*>(smem + L::kRing + w * L::kSlotBytes);
        };
        float2 ml[kStreamWarps];
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kStreamWarps; ++w) {
            ml[w] = ((mask >> w) & 1u) ? reinterpret_cast<const float2*>(piece(w) + ROWS * L::kSlotRow)[r]
                                       : make_float2(-INFINITY, 0.f);
            M = fmaxf(M, ml[w].x);
        }
        float lsum = 0.f, acc[kPer];
#pragma unroll
        for (int c = 0; c < kPer; ++c) acc[c] = 0.f;
#pragma unroll
        for (int w = 0; w < kStreamWarps; ++w) {
            if (!((mask >> w) & 1u)) continue;
            const float wt = ml[w].x == -INFINITY ? 0.f : fast_exp2(ml[w].x - M);
            lsum += wt * ml[w].y;
            const float* src = piece(w) + r * L::kSlotRow + lane * kPer;
            if constexpr (kPer == 4) {
                const float4 v = *reinterpret_cast<const float4*>(src);
                acc[0] += wt * v.x;
                acc[1] += wt * v.y;
                acc[2] += wt * v.z;
                acc[3] += wt * v.w;
            } else {
                const float2 v = *reinterpret_cast<const float2*>(src);
                acc[0] += wt * v.x;
                acc[1] += wt * v.y;
            }
        }
        if (t.x < 0) {
            const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
            uint16_t* dst = out + ((long)(h.x + r / g) * Hq + h.y * g + r % g) * D + lane * kPer;
            if constexpr (kPer == 4)
                *reinterpret_cast<uint2*>(dst) =
                    make_uint2(pack_bf16x2(acc[0] * inv, acc[1] * inv), pack_bf16x2(acc[2] * inv, acc[3] * inv));
            else
                *reinterpret_cast<uint32_t*>(dst) = pack_bf16x2(acc[0] * inv, acc[1] * inv);
        } else {
            float* dst = part_o + ((long)t.x * kDecodeRows + r) * D + lane * kPer;
            if constexpr (kPer == 4)
                *reinterpret_cast<float4*>(dst) = make_float4(acc[0], acc[1], acc[2], acc[3]);
            else
                *reinterpret_cast<float2*>(dst) = make_float2(acc[0], acc[1]);
            if (lane == 0) part_ml[(long)t.x * kDecodeRows + r] = make_float2(M, lsum);
        }
    }
}

// Merges the partials of segments cut by the decode CTAs' range boundaries (one
// piece per CTA, the CTA having combined its warps' pieces already): for row
// r, m = max_p m_p, l = sum_p 2^(m_p - m) l_p, O = sum_p 2^(m_p - m) O_p / l
// (base 2, O_p unnormalised).  One CTA per (sequence, kv head) with one warp
// per output row (as many warps as the batch's longest decode chunk has rows):
// lane j owns channels 4j..4j+3 and piece j's statistics.  The first four
// pieces' O rows are requested together with the statistics, the rest eight
// (then four) at a time, so a segment cut into few pieces costs one round
// trip.  The programmatic launch lets the CTAs compute their offsets as decode
// CTAs exit; they read partials only after griddepcontrol.wait.
constexpr int kMergeMaxThreads = 32 * kDecodeRows;
template <int D>
__global__ void __launch_bounds__(kMergeMaxThreads, 1) paged_merge_kernel(const int32_t* __restrict__ ctx_lens,
                                                                    const int32_t* __restrict__ q_lens,
                                                                    const float* part_o, const float2* part_ml,
                                                                    uint16_t* __restrict__ out, int num_seqs,
                                                                    int Hq, int Hkv, int mbps, int W) {
    // one warp per output row: warp w of CTA (s, hk) merges row w
    const int s = blockIdx.x, hk = blockIdx.y, r = threadIdx.x >> 5, g = Hq / Hkv;
    const int lane = threadIdx.x & 31;
    const int ql_s = __ldg(q_lens + s), cl_s = __ldg(ctx_lens + s);
    const bool mine = is_decode_row(ql_s, g) && ql_s <= cl_s && cl_s <= mbps * kBS && r < g * ql_s;
    if (!mine) {
        // every CTA waits for the decode grid, so this grid never completes ahead of it
        asm volatile("griddepcontrol.wait;" ::: "memory");
        return;
    }
    const int nblk = (cl_s + kBS - 1) / kBS;
    // inputs only so far: total pages, this sequence's first page and query row
    long long tot = 0, pre = 0, q0 = 0;
    for (int i = lane; i < num_seqs; i += 32) {
        const int ql = __ldg(q_lens + i), cl = __ldg(ctx_lens + i);
        const long long n = (is_decode_row(ql, g) && ql <= cl && cl <= mbps * kBS) ? (cl + kBS - 1) / kBS : 0;
        tot += n;
        if (i < s) {
            pre += n;
            q0 += ql;
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        tot += __shfl_xor_sync(0xffffffffu, tot, o);
        pre += __shfl_xor_sync(0xffffffffu, pre, o);
        q0 += __shfl_xor_sync(0xffffffffu, q0, o);
    }
    const long long P = (long long)Hkv * tot;
    const long long seg_first = (long long)Hkv * pre + (long long)hk * nblk;
    const StreamSplit split(P, W);  // W: the decode grid's warps
    const int c_lo = split.owner(seg_first) / kStreamWarps, c_hi = split.owner(seg_first + nblk - 1) / kStreamWarps;
    const int npieces = c_hi - c_lo + 1;
    // slot of piece k: 2c, or 2c+1 when the segment starts after CTA c's first
    // page; -1 when CTA c's range is empty (fewer pages than warps: it wrote nothing)
    auto slot_of = [&](int k) -> long {
        const int c = c_lo + k;
        const long long cb = split.begin(c * kStreamWarps);
        if (split.begin((c + 1) * kStreamWarps) == cb) return -1;
        return 2L * c + (seg_first <= cb ? 0 : 1);
    };
    const long lane_slot = lane < npieces ? slot_of(lane) : -1;
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (c_lo == c_hi) return;  // the whole segment was finished inside one decode CTA

    constexpr int kPer = D / 32;  // channels per lane
    float acc[kPer];
#pragma unroll
    for (int c = 0; c < kPer; ++c) acc[c] = 0.f;
    float lsum = 0.f, M = -INFINITY;
    // pieces in groups of 32: lane j holds piece j's (max, sum); the running
    // max of earlier groups rescales the accumulators
    for (int c0 = 0; c0 < npieces; c0 += 32) {
        const long myslot = c0 + lane < npieces ? (c0 == 0 ? lane_slot : slot_of(c0 + lane)) : -1;
        const int n = min(32, npieces - c0);
        // partials are read through L2 (ld.global.cg): the decode grid wrote them
        // while this grid was already resident, so the read-only path is not valid.
        // The first four pieces' O rows do not depend on the statistics: requested with them.
        float v0[4][kPer];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const long sj = __shfl_sync(0xffffffffu, myslot, u);
            if (u < n && sj >= 0) {
                const float* src = part_o + (sj * kDecodeRows + r) * D + lane * kPer;
                if constexpr (kPer == 4) {
                    const float4 t4 = __ldcg(reinterpret_cast<const float4*>(src));
                    v0[u][0] = t4.x; v0[u][1] = t4.y; v0[u][2] = t4.z; v0[u][3] = t4.w;
                } else {
                    const float2 t2 = __ldcg(reinterpret_cast<const float2*>(src));
                    v0[u][0] = t2.x; v0[u][1] = t2.y;
                }
            } else {
#pragma unroll
                for (int c = 0; c < kPer; ++c) v0[u][c] = 0.f;
            }
        }
        const float2 ml = myslot >= 0 ? __ldcg(part_ml + myslot * kDecodeRows + r) : make_float2(-INFINITY, 0.f);
        float gm = ml.x;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) gm = fmaxf(gm, __shfl_xor_sync(0xffffffffu, gm, o));
        const float Mn = fmaxf(M, gm);
        if (Mn == -INFINITY) continue;  // nothing visible yet (uniform)
        const float rescale = M == -INFINITY ? 0.f : fast_exp2(M - Mn);
#pragma unroll
        for (int c = 0; c < kPer; ++c) acc[c] *= rescale;
        lsum *= rescale;
        M = Mn;
        const float w = myslot >= 0 ? fast_exp2(ml.x - M) : 0.f;
        lsum += w * ml.y;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const float wu = __shfl_sync(0xffffffffu, w, u);  // 0 past the group or for an empty range
#pragma unroll
            for (int c = 0; c < kPer; ++c) acc[c] += wu * v0[u][c];
        }
        int j = 4;
        for (; j + 8 <= n; j += 8) {  // eight pieces' loads in flight at once
            float v[8][kPer];
            float wj[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                wj[u] = __shfl_sync(0xffffffffu, w, j + u);
                const long sj = __shfl_sync(0xffffffffu, myslot, j + u);
                const float* src = part_o + ((sj < 0 ? 0 : sj) * kDecodeRows + r) * D + lane * kPer;
                if constexpr (kPer == 4) {
                    const float4 t = __ldcg(reinterpret_cast<const float4*>(src));
                    v[u][0] = t.x; v[u][1] = t.y; v[u][2] = t.z; v[u][3] = t.w;
                } else {
                    const float2 t = __ldcg(reinterpret_cast<const float2*>(src));
                    v[u][0] = t.x; v[u][1] = t.y;
                }
                if (sj < 0)  // an empty range wrote no partial: ignore whatever the slot holds
#pragma unroll
                    for (int c = 0; c < kPer; ++c) v[u][c] = 0.f;
            }
#pragma unroll
            for (int u = 0; u < 8; ++u)
#pragma unroll
                for (int c = 0; c < kPer; ++c) acc[c] += wj[u] * v[u][c];
        }
        for (; j < n; j += 4) {  // the rest, four pieces' loads in flight at once
            float v[4][kPer];
            float wj[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int k = j + u;
                wj[u] = __shfl_sync(0xffffffffu, w, k & 31);
                const long sj = __shfl_sync(0xffffffffu, myslot, k & 31);
                if (k < n && sj >= 0) {
                    const float* src = part_o + (sj * kDecodeRows + r) * D + lane * kPer;
                    if constexpr (kPer == 4) {
                        const float4 t4 = __ldcg(reinterpret_cast<const float4*>(src));
                        v[u][0] = t4.x; v[u][1] = t4.y; v[u][2] = t4.z; v[u][3] = t4.w;
                    } else {
                        const float2 t2 = __ldcg(reinterpret_cast<const float2*>(src));
                        v[u][0] = t2.x; v[u][1] = t2.y;
                    }
                } else {
                    wj[u] = 0.f;
#pragma unroll
                    for (int c = 0; c < kPer; ++c) v[u][c] = 0.f;
                }
            }
#pragma unroll
            for (int u = 0; u < 4; ++u)
#pragma unroll
                for (int c = 0; c < kPer; ++c) acc[c] += wj[u] * v[u][c];
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) lsum += __shfl_xor_sync(0xffffffffu, lsum, o);
    const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
    uint16_t* dst = out + ((long)(q0 + r / g) * Hq + hk * g + r % g) * D + lane * kPer;
    if constexpr (kPer == 4)
        *reinterpret_cast<uint2*>(dst) =
            make_uint2(pack_bf16x2(acc[0] * inv, acc[1] * inv), pack_bf16x2(acc[2] * inv, acc[3] * inv));
    else
        *reinterpret_cast<uint32_t*>(dst) = pack_bf16x2(acc[0] * inv, acc[1] * inv);
}

// ------------------------------------------------------------ metadata -----
// One CTA: q_start (exclusive prefix sum of q_lens) and the list of work
// entries (entry_tokens consecutive query tokens, paged_tc_entry_tokens) of
// the sequences that take the tensor-core kernel, ordered by decreasing number
// of KV tiles (longest first) with a counting sort.  Entry = (sequence, first
// query token of the entry within the chunk).
__global__ void __launch_bounds__(1024) paged_meta_kernel(const int32_t* __restrict__ ctx_lens,
                                                          const int32_t* __restrict__ q_lens, int num_seqs, int mbps,
                                                          int g, int causal, int entry_tokens,
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
        const int last_row = min(ql, t0 + entry_tokens) - 1;  // last query row of the entry
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
        for (int t0 = 0; t0 < ql; t0 += entry_tokens) atomicAdd(&hist[entry_cost(ql, cl, t0)], 1);
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
        count[1] = 0;  // the tensor-core kernel's unit tickets
    }
    __syncthreads();
    for (int s = threadIdx.x; s < num_seqs; s += blockDim.x) {
        const int ql = q_lens[s], cl = ctx_lens[s];
        if (ql <= 0 || is_decode_row(ql, g) || ql > cl || cl > mbps * kBS) continue;
        for (int t0 = 0; t0 < ql; t0 += entry_tokens) {
            const int pos = atomicAdd(&hist[entry_cost(ql, cl, t0)], 1);
            if (pos < max_entries) {
                list[2 * pos] = s;
                list[2 * pos + 1] = t0;
            }
        }
    }
}

// A library-owned side stream per device: the chunked-prefill metadata pass (one
// CTA) runs there beside the split-KV decode kernel and its merge, which do
// not depend on it; two events fork it from and join it back to the caller's
// stream (both capturable, so the call may be recorded into a CUDA graph).
constexpr int kMaxSideDevices = 64;
struct SideStream {
    std::mutex mu;
    cudaStream_t s = nullptr;
    cudaEvent_t fork = nullptr, join = nullptr;
};
SideStream g_side[kMaxSideDevices];

static fa_status side_stream(SideStream** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxSideDevices) return FA_ERR_CUDA;
    SideStream& ss = g_side[dev];
    if (!ss.s && cudaStreamCreateWithFlags(&ss.s, cudaStreamNonBlocking) != cudaSuccess) return FA_ERR_CUDA;
    if (!ss.fork && cudaEventCreateWithFlags(&ss.fork, cudaEventDisableTiming) != cudaSuccess) return FA_ERR_CUDA;
    if (!ss.join && cudaEventCreateWithFlags(&ss.join, cudaEventDisableTiming) != cudaSuccess) return FA_ERR_CUDA;
    *out = &ss;
    return FA_OK;
}

template <int D, bool KV8 = false>
static fa_status launch_decode(const void* q, const void* k_cache, const void* v_cache, const int32_t* bt,
                               const int32_t* ctx_lens, const int32_t* q_lens, void* out, const PagedWs& w,
                               uint8_t* ws, int num_seqs, int mbps, int num_blocks, int Hq, int Hkv,
                               int q_prefetch_rows, int causal, float scale, int merge_rows, cudaStream_t s,
                               const DevCtx& ctx, int* launches,
                               float k_scale = 1.f, float v_scale = 1.f) {
    CUtensorMap tk, tv;
    fa_status st;
    if constexpr (KV8) {
        // K [blocks][Hkv][16][D] bytes, rows of D bytes, 128-byte swizzle;
        // V [blocks][Hkv][D][16] bytes, one 16-byte row per channel
        const uint64_t kd[4] = {(uint64_t)D, (uint64_t)kBS, (uint64_t)Hkv, (uint64_t)num_blocks};
        const uint64_t vd[4] = {(uint64_t)kBS, (uint64_t)D, (uint64_t)Hkv, (uint64_t)num_blocks};
        const uint64_t ks[3] = {(uint64_t)D, (uint64_t)kBS * D, (uint64_t)Hkv * kBS * D};
        const uint64_t vs[3] = {(uint64_t)kBS, (uint64_t)kBS * D, (uint64_t)Hkv * kBS * D};
        const uint32_t kb[4] = {(uint32_t)D, (uint32_t)kBS, 1, 1};
        const uint32_t vb[4] = {(uint32_t)kBS, (uint32_t)D, 1, 1};
        st = encode_tmap_4d(&tk, k_cache, kd, ks, kb, CU_TENSOR_MAP_DATA_TYPE_UINT8, CU_TENSOR_MAP_SWIZZLE_128B);
        if (st != FA_OK) return st;
        st = encode_tmap_4d(&tv, v_cache, vd, vs, vb, CU_TENSOR_MAP_DATA_TYPE_UINT8, CU_TENSOR_MAP_SWIZZLE_NONE);
        if (st != FA_OK) return st;
    } else {
        const uint64_t dims[4] = {(uint64_t)D, (uint64_t)kBS, (uint64_t)Hkv, (uint64_t)num_blocks};
        const uint64_t strides[3] = {(uint64_t)D * 2, (uint64_t)kBS * D * 2, (uint64_t)Hkv * kBS * D * 2};
        const uint32_t box[4] = {64, (uint32_t)kBS, 1, 1};
        st = encode_tmap_bf16_4d(&tk, k_cache, dims, strides, box);
        if (st != FA_OK) return st;
        if ((st = encode_tmap_bf16_4d(&tv, v_cache, dims, strides, box)) != FA_OK) return st;
    }
    float* part_o = reinterpret_cast<float*>(ws + w.part_o);
    float2* part_ml = reinterpret_cast<float2*>(ws + w.part_ml);
    const float scale_log2 = scale * k_scale * 1.4426950408889634f;
    const int grid = std::min(sm_count(), kMaxStreamCtas);
    // partial slots of 6 rows when no decode chunk has more (then the ring keeps
    // three stages at d = 128), else of 16
    auto launch = [&](auto rows) -> fa_status {
        constexpr int R = decltype(rows)::value;
        using L = StreamSmem<D, KV8, R>;
        const fa_status st2 = raise_dynamic_smem(reinterpret_cast<const void*>(paged_decode_kernel<D, KV8, R>), L::kBytes);
        if (st2 != FA_OK) return st2;
        paged_decode_kernel<D, KV8, R><<<grid, kStreamWarps * 32, L::kBytes, s>>>(
            tk, tv, static_cast<const uint16_t*>(q), bt, ctx_lens, q_lens, static_cast<uint16_t*>(out), part_o, part_ml,
            num_seqs, mbps, num_blocks, Hq, Hkv, q_prefetch_rows, causal, scale_log2, v_scale, ctx);
        return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
    };
    st = merge_rows <= 6 ? launch(std::integral_constant<int, 6>{}) : launch(std::integral_constant<int, kDecodeRows>{});
    if (st != FA_OK) return st;
    ++*launches;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(num_seqs, Hkv, 1);
    cfg.blockDim = dim3(32 * merge_rows);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, paged_merge_kernel<D>, ctx_lens, q_lens, static_cast<const float*>(part_o),
                           static_cast<const float2*>(part_ml), static_cast<uint16_t*>(out), num_seqs, Hq, Hkv,
                           mbps, grid * kStreamWarps) != cudaSuccess)
        return FA_ERR_CUDA;
    ++*launches;
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
    const bool decode_path = g <= kDecodeRows;  // some sequences may be decode rows
    const bool tc_path = !is_decode_row(max_q_len, g);
    // the tensor-core path's work list: on the side stream when the decode
    // kernel also runs (they are independent), else in line
    SideStream* ss = nullptr;
    std::unique_lock<std::mutex> side_lock;
    if (tc_path) {
        const int entry_tokens = paged_tc_entry_tokens(g);
        int32_t* q_start = reinterpret_cast<int32_t*>(wsb + w.q_start);
        int32_t* count = reinterpret_cast<int32_t*>(wsb + w.work_count);
        int32_t* list = reinterpret_cast<int32_t*>(wsb + w.work_list);
        const int nbins = (max_blocks_per_seq * kBS + 127) / 128 + 1;
        const size_t hist_bytes = sizeof(int) * (size_t)(nbins + 1);
        if (hist_bytes > 200 * 1024) return FA_ERR_UNSUPPORTED;
        if (hist_bytes > 48 * 1024 &&
            (st = raise_dynamic_smem(reinterpret_cast<const void*>(paged_meta_kernel), (int)hist_bytes)) != FA_OK)
            return st;
        cudaStream_t ms = s;
        if (decode_path) {
            if ((st = side_stream(&ss)) != FA_OK) return st;
            side_lock = std::unique_lock<std::mutex>(ss->mu);
            if (cudaEventRecord(ss->fork, s) != cudaSuccess || cudaStreamWaitEvent(ss->s, ss->fork, 0) != cudaSuccess)
                return FA_ERR_CUDA;
            ms = ss->s;
        }
        paged_meta_kernel<<<1, 1024, hist_bytes, ms>>>(ctx_lens, q_lens, num_seqs, max_blocks_per_seq, g, causal,
                                                       entry_tokens, q_start, count, list, w.max_entries, ctx);
        const bool launched = cudaGetLastError() == cudaSuccess;
        if (ss && (cudaEventRecord(ss->join, ss->s) != cudaSuccess || !launched)) {
            (void)cudaStreamWaitEvent(s, ss->join, 0);  // leave the side stream joined
            return FA_ERR_CUDA;
        }
        if (!launched) return FA_ERR_CUDA;
        ++launches;
    }
    if (decode_path) {
        const int merge_rows = (int)std::min<long>(kDecodeRows, (long)g * max_q_len);
        const int qpf = is_decode_row(max_q_len, g) ? total_q : 0;  // every query row is a decode row
        st = d == 128 ? launch_decode<128>(q, k_cache, v_cache, block_table, ctx_lens, q_lens, out, w, wsb, num_seqs,
                                           max_blocks_per_seq, num_blocks, Hq, Hkv, qpf, causal, scale, merge_rows, s,
                                           ctx, &launches)
                      : launch_decode<64>(q, k_cache, v_cache, block_table, ctx_lens, q_lens, out, w, wsb, num_seqs,
                                          max_blocks_per_seq, num_blocks, Hq, Hkv, qpf, causal, scale, merge_rows, s,
                                          ctx, &launches);
        if (st != FA_OK) {
            if (ss) (void)cudaStreamWaitEvent(s, ss->join, 0);  // keep the side stream joined
            return st;
        }
    }
    if (tc_path) {
        if (ss && cudaStreamWaitEvent(s, ss->join, 0) != cudaSuccess) return FA_ERR_CUDA;
        int32_t* q_start = reinterpret_cast<int32_t*>(wsb + w.q_start);
        int32_t* count = reinterpret_cast<int32_t*>(wsb + w.work_count);
        int32_t* list = reinterpret_cast<int32_t*>(wsb + w.work_list);
        st = launch_paged_prefill(q, k_cache, v_cache, block_table, ctx_lens, q_lens, q_start, list, count, out,
                                  num_seqs, max_blocks_per_seq, num_blocks, Hq, Hkv, d, causal, scale, total_q, s,
                                  ctx);
        if (st != FA_OK) return st;
        ++launches;
    }
    set_launch_count(launches);
    return FA_OK;
}

fa_status fa_paged_attn_fp8(const void* q, const void* k_cache, const void* v_cache, float k_scale, float v_scale,
                            const int32_t* block_table, const int32_t* ctx_lens, const int32_t* q_lens, void* out,
                            int num_seqs, int max_blocks_per_seq, int num_blocks, int Hq, int Hkv, int d,
                            int block_size, int causal, float scale, int total_q, int max_q_len, void* ws,
                            size_t ws_bytes, fa_stream_t stream) {
    set_launch_count(0);
    if (num_seqs < 0 || max_blocks_per_seq < 0 || num_blocks < 0 || Hq <= 0 || Hkv <= 0 || total_q < 0 ||
        max_q_len < 0 || !(scale > 0.f) || !(scale < INFINITY) || !(k_scale > 0.f) || !(k_scale < INFINITY) ||
        !(v_scale > 0.f) || !(v_scale < INFINITY))
        return FA_ERR_INVALID_ARG;
    if (block_size != kBS || d != 128 || Hq % Hkv != 0) return FA_ERR_UNSUPPORTED;
    if (num_seqs == 0 || total_q == 0 || max_q_len == 0) return FA_OK;
    if (!is_decode_row(max_q_len, Hq / Hkv)) return FA_ERR_UNSUPPORTED;  // decode rows only
    if (!q || !k_cache || !v_cache || !block_table || !ctx_lens || !q_lens || !out) return FA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned32(out)) return FA_ERR_INVALID_ARG;
    if (num_blocks == 0 || max_blocks_per_seq == 0) return FA_ERR_INVALID_ARG;
    const PagedWs w = paged_ws_layout(num_seqs, max_blocks_per_seq, Hq, Hkv, d, total_q);
    if (!ws || ws_bytes < w.total || (reinterpret_cast<uintptr_t>(ws) & 255)) return FA_ERR_WORKSPACE;
    fa_status st = check_device();
    if (st != FA_OK) return st;
    DevCtx ctx;
    if ((st = make_ctx(&ctx)) != FA_OK) return st;
    int launches = 0;
    st = launch_decode<128, true>(q, k_cache, v_cache, block_table, ctx_lens, q_lens, out, w,
                                  static_cast<uint8_t*>(ws), num_seqs, max_blocks_per_seq, num_blocks, Hq, Hkv,
                                  total_q, causal, scale, (Hq / Hkv) * max_q_len,
                                  reinterpret_cast<cudaStream_t>(stream), ctx, &launches, k_scale, v_scale);
    if (st != FA_OK) return st;
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
