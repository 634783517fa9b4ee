// Tensor-core attention for sm_103a: the tiled online-softmax algorithm of
// "Fast Attention Kernels and Operator Fusion", section "FlashAttention-Style
// Kernels" (queries, keys and values processed in tiles; per tile a block of
// scores, an update of the softmax statistics and an on-chip accumulation of
// the output; the score matrix never stored in device memory), for
//   * contiguous prefill        (MODE_DENSE),
//   * prefill with an additive mask M, classified per 128x128 tile beforehand
//     (tiles of -inf skipped; tiles of 0 read no mask; tiles of 0 and -inf
//     that keep one run of keys per row apply that run like the causal limit;
//     other tiles add M)        (MODE_MASKED),
//   * chunked prefill over the paged cache, every K/V tile gathered block by
//     block through the block table, one copy per 16-token block (MODE_PAGED;
//     section "Paged Attention Kernels").
//
// CTA layout (320 threads, one CTA per SM, persistent over work units):
//   warps 0-3   softmax warpgroup of Q slot 0, warps 4-7 of Q slot 1: thread
//               r owns query row r of its slot (TMEM lane r; warp w may only
//               touch TMEM lanes 32*(w%4) .. 32*(w%4)+31);
//   warp 8      TMA producer: Q tiles once per unit, then K_j, V_j into a ring
//               of shared-memory stages (128-byte swizzle);
//   warp 9      tcgen05.mma issuer (one thread) and TMEM owner.
// A work unit is two 128-row Q tiles ("slots") that share one kv head: two
// query heads of the same GQA group over the same rows when Hq/Hkv is even,
// otherwise two consecutive row tiles of one head.  Both slots consume the
// same K/V tiles, so K/V are staged once for two Q tiles.
//
// TMEM (512 columns x 128 lanes, fp32): S0 [0,128), S1 [128,256),
// O0 [256, 256+d), O1 [256+d, 256+2d).  P (bf16, packed two per column) is
// written by the softmax threads over the first 64 columns of S and fed to
// the P*V MMA straight from TMEM.
//
// MMA order per KV tile j:  PV0(j-1), QK0(j), PV1(j-1), QK1(j).  Each
// tcgen05.commit tracks every MMA issued before it, so when slot s sees S_s(j)
// complete, PV_s(j-1) is complete too and O_s may be rescaled.
//
// Softmax: base-2 exponentials with scale*log2(e) folded in; the running max
// is only moved when a row's max grows by more than 8 (a factor 256), so O and
// the row sum stay consistent with a possibly stale max (exact up to
// rounding); P is rounded to bf16 for the tensor core, row sums stay fp32.
#include <algorithm>
#include <cmath>

#include <memory>
#include <mutex>
#include <vector>

#include "host_common.cuh"

namespace fa {

enum { MODE_DENSE = 0, MODE_MASKED = 1, MODE_PAGED = 2 };
constexpr int kRangeHoles = 1 << 30;  // flag bit of a query tile's visible KV range
constexpr int kTcThreads = 320;
constexpr int kProducerWarp = 8, kMmaWarp = 9;
constexpr int kTcRows = 128;  // rows of a Q tile and of a KV tile
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;
// Paged mode hands out work units at run time: the producer takes a ticket
// from a counter in the workspace (zeroed by the metadata kernel before every
// launch) when it starts a unit, and passes the unit to the MMA and softmax
// warps through a ring of kUnitSlots mailboxes.
constexpr int kUnitSlots = 4;
constexpr int kUnitReaders = 9;  // the MMA warp and the eight softmax warps

template <int D>
struct TcCfg {
    static constexpr int kAtoms = D / 64;                 // 128-byte column blocks per row
    static constexpr int kAtomBytes = kTcRows * 128;      // one 128-row x 64-channel box
    static constexpr int kTileBytes = kAtoms * kAtomBytes;
    static constexpr int kStages = D == 128 ? 5 : 8;
    static constexpr int kQBytes = 2 * kTileBytes;
    static constexpr int kRingBytes = kStages * kTileBytes;
    static constexpr int kNumBars = 2 * kStages + 2 * 6 + 2 + 2 * kUnitSlots;
    static constexpr int kSmem = 1024 + kQBytes + kRingBytes + kNumBars * 8 + 16 + 4 * kUnitSlots;
    static constexpr uint32_t kS0 = 0, kS1 = 128, kO0 = 256, kO1 = 256 + D;
    // Paged K/V tiles hold each 8-row group's 64-channel halves side by side
    // ([group][half][8 rows][128 B]), so that one copy lands a whole 16-token
    // block: 8-row groups kPagedGroup bytes apart, halves 1024 bytes apart.
    // Dense tiles hold one half after the other ([half][128 rows][128 B]).
    static constexpr uint32_t kPagedGroup = kAtoms * 1024;
};

struct TcParams {
    int B, T;        // dense / masked: sequence length (row stride of q/k/v/out)
    int q0, Tq, Tk;  // dense: query rows [q0, q0 + Tq) of each sequence against keys [0, Tk)
                     // (q0 a multiple of 128; q0 = 0, Tq = Tk = T for the whole problem)
    int Hq, Hkv, g;
    int causal;
    float scale_log2;
    int pair_heads;  // 1: slots = heads (2pp, 2pp+1) of a group; 0: row tiles (2t, 2t+1) of one head
    int pack;        // paged: a slot is 128/g tokens x the g heads of a group (row = token * g + head)
    int pack_shift;  // log2(g) when packed
    int num_units;   // dense / masked
    uint16_t* out;
    float* lse;
    // masked
    const float* mask;
    const uint8_t* cls;
    const uint8_t* iv;  // per tile: 128 rows x (lo, hi), the run of keys a class-3 tile keeps
    const int32_t* qt_order;
    const int2* qt_range;  // per query tile: [first, last+1) of its KV tiles that are not all -inf;
                           // kRangeHoles set in .x when an all -inf tile lies inside that range
    // paged
    const int32_t* bt;
    const int32_t* ctx_lens;
    const int32_t* q_lens;
    const int32_t* q_start;
    const int32_t* work_list;
    const int32_t* work_count;
    int mbps, num_blocks;
    DevCtx ctx;
};

struct Unit {
    int b;          // batch (dense) / sequence (paged)
    int hk;         // kv head
    int head[2];    // query head per slot
    int row0[2];    // first query row per slot (within T, or within the chunk)
    int nrows[2];   // valid rows per slot (0: slot idle)
    int qtok[2];    // row coordinate for the Q tile load
    int kv_len;     // keys of the sequence (T or ctx)
    int pos_off;    // key position of query row i is i + pos_off
    int kt0;        // first KV tile to scan
    int n_kt;       // KV tiles to scan: [kt0, n_kt)
    int holes;      // masked: some tile in [kt0, n_kt) is all -inf for both slots (must be skipped)
};

// Per-slot field of a unit.  A select instead of a runtime array index keeps
// the value in a register (a runtime index would move the array to local memory).
__device__ __forceinline__ int sel(const int (&a)[2], int s) { return s ? a[1] : a[0]; }

// i-th unit of this CTA: units are ordered longest first and dealt to the CTAs
// in boustrophedon order (round i goes left to right when even, right to left
// when odd), which evens out the per-CTA totals.
__device__ __forceinline__ int unit_of(int i, int G) {
    const int c = blockIdx.x;
    return i * G + ((i & 1) ? (G - 1 - c) : c);
}

// An explicit unit-to-CTA assignment computed on the host (dense causal
// prefill, where every unit's cost is known there): CTA c runs units
// unit[start[c] .. start[c+1]).  Passed by value as a kernel parameter, so
// it needs no device memory and a captured graph keeps it.  n == 0: use
// unit_of.
constexpr int kMaxSchedCtas = 160;
constexpr int kMaxSchedUnits = 2048;
struct TcSched {
    int n;
    uint16_t start[kMaxSchedCtas + 1];
    uint16_t unit[kMaxSchedUnits];
};

// This CTA's i-th unit, or -1 after its last one.
__device__ __forceinline__ int cta_unit(const TcSched& sc, int i, int G, int num_units) {
    if (sc.n > 0) {
        const int k = sc.start[blockIdx.x] + i;
        return k < sc.start[blockIdx.x + 1] ? (int)sc.unit[k] : -1;
    }
    if (i * G >= num_units) return -1;
    const int u = unit_of(i, G);
    return u < num_units ? u : -1;
}

// Units of one paged work entry: one per kv head (packed), per head pair, or per head.
__device__ __forceinline__ int paged_units_per_entry(const TcParams& p) {
    return p.pack ? p.Hkv : (p.pair_heads ? p.Hkv * (p.g / 2) : p.Hq);
}

template <int MODE>
__device__ __forceinline__ Unit decode_unit(const TcParams& p, int u) {
    Unit U;
    U.holes = 0;
    if constexpr (MODE == MODE_PAGED) {
        const int per_entry = paged_units_per_entry(p);
        const int e = u / per_entry, rest = u % per_entry;
        const int seq = __ldg(p.work_list + 2 * e), t0 = __ldg(p.work_list + 2 * e + 1);
        const int ql = __ldg(p.q_lens + seq), cl = __ldg(p.ctx_lens + seq), qs = __ldg(p.q_start + seq);
        U.b = seq;
        int slot_tokens = kTcRows;
        if (p.pack) {  // all heads of kv head `rest`'s group, two blocks of 128/g tokens
            slot_tokens = kTcRows >> p.pack_shift;
            U.hk = rest;
            U.head[0] = U.head[1] = rest * p.g;  // first head of the group
            U.row0[0] = t0;
            U.row0[1] = t0 + slot_tokens;
        } else if (p.pair_heads) {
            const int pp = rest % (p.g / 2);
            U.hk = rest / (p.g / 2);
            U.head[0] = U.hk * p.g + 2 * pp;
            U.head[1] = U.head[0] + 1;
            U.row0[0] = U.row0[1] = t0;
        } else {
            U.head[0] = U.head[1] = rest;
            U.hk = rest / p.g;
            U.row0[0] = t0;
            U.row0[1] = t0 + kTcRows;
        }
        int last = 0;
#pragma unroll
        for (int s = 0; s < 2; ++s) {
            U.nrows[s] = max(0, min(slot_tokens, ql - U.row0[s]));  // query tokens of the slot
            U.qtok[s] = qs + U.row0[s];
            if (U.nrows[s] > 0) last = max(last, U.row0[s] + U.nrows[s]);
        }
        U.kv_len = cl;
        U.pos_off = cl - ql;
        const int kv_end = p.causal ? min(cl, cl - ql + last) : cl;
        U.kt0 = 0;
        U.n_kt = (kv_end + kTcRows - 1) / kTcRows;
    } else {
        const int nqt = (p.Tq + kTcRows - 1) / kTcRows;  // query tiles of this launch
        const int qt0 = p.q0 / kTcRows;                  // its first tile within the sequence
        if (p.pair_heads) {
            const int half = p.g / 2;
            const int upt = p.B * p.Hkv * half;
            const int rank = u / upt, rest = u % upt;
            int qt;
            if constexpr (MODE == MODE_MASKED)
                qt = __ldg(p.qt_order + rank);
            else
                qt = p.causal ? nqt - 1 - rank : rank;
            U.b = rest / (p.Hkv * half);
            U.hk = (rest / half) % p.Hkv;
            const int pp = rest % half;
            U.head[0] = U.hk * p.g + 2 * pp;
            U.head[1] = U.head[0] + 1;
            U.row0[0] = U.row0[1] = (qt0 + qt) * kTcRows;
        } else {
            const int ntp = (nqt + 1) / 2;
            const int upt = p.B * p.Hq;
            const int rank = u / upt, rest = u % upt;
            const int pt = (p.causal && MODE == MODE_DENSE) ? ntp - 1 - rank : rank;
            U.b = rest / p.Hq;
            U.head[0] = U.head[1] = rest % p.Hq;
            U.hk = U.head[0] / p.g;
            U.row0[0] = (qt0 + 2 * pt) * kTcRows;
            U.row0[1] = (qt0 + 2 * pt + 1) * kTcRows;
        }
        int last = 0;
#pragma unroll
        for (int s = 0; s < 2; ++s) {
            U.nrows[s] = max(0, min(kTcRows, p.q0 + p.Tq - U.row0[s]));
            U.qtok[s] = U.row0[s];
            if (U.nrows[s] > 0) last = max(last, U.row0[s] + U.nrows[s]);
        }
        U.kv_len = p.Tk;
        U.pos_off = 0;  // rows and keys are both absolute positions in the sequence
        const int kv_end = p.causal ? min(p.Tk, last) : p.Tk;
        U.kt0 = 0;
        U.n_kt = (kv_end + kTcRows - 1) / kTcRows;
        if constexpr (MODE == MODE_MASKED) {
            // restrict the scan to the KV tiles the mask leaves visible; the
            // tiles inside that range need a per-tile class check only when
            // one of them is all -inf for both slots (a hole in a slot's range,
            // or a gap between the two slots' ranges)
            int lo = U.n_kt, hi = 0, lo_s[2] = {0, 0}, hi_s[2] = {0, 0}, live = 0;
#pragma unroll
            for (int s = 0; s < 2; ++s)
                if (U.nrows[s] > 0) {
                    const int2 r = __ldg(p.qt_range + U.row0[s] / kTcRows);
                    const int rlo = r.x & (kRangeHoles - 1);
                    lo_s[s] = rlo;
                    hi_s[s] = r.y;
                    lo = min(lo, rlo);
                    hi = max(hi, r.y);
                    U.holes |= (r.x & kRangeHoles) ? 1 : 0;
                    ++live;
                }
            if (live == 2 && (hi_s[0] < lo_s[1] || hi_s[1] < lo_s[0])) U.holes = 1;
            U.kt0 = lo;
            U.n_kt = min(U.n_kt, hi);
        }
    }
    return U;
}

// Mask class of (query tile of slot s, KV tile kt): 0 skip, 1 no mask, 2 mixed.
template <int MODE>
__device__ __forceinline__ int tile_class(const TcParams& p, const Unit& U, int s, int kt) {
    if constexpr (MODE == MODE_MASKED) {
        if (sel(U.nrows, s) <= 0) return 0;
        const int nkt = (p.T + kTcRows - 1) / kTcRows;
        return __ldg(p.cls + (long)(sel(U.row0, s) / kTcRows) * nkt + kt);
    } else {
        return sel(U.nrows, s) > 0 ? 1 : 0;
    }
}

template <int MODE>
__device__ __forceinline__ bool skip_tile(const TcParams& p, const Unit& U, int kt) {
    if constexpr (MODE == MODE_MASKED)
        return U.holes && tile_class<MODE>(p, U, 0, kt) == 0 && tile_class<MODE>(p, U, 1, kt) == 0;
    else
        return false;
}

template <int MODE>
__device__ __forceinline__ bool unit_active(const TcParams& p, const Unit& U) {
    (void)p;
    return U.kt0 < U.n_kt;  // in masked mode [kt0, n_kt) starts and ends on a visible tile
}

// Output row of slot s of a unit (bf16, d channels): query token `tok` of the
// slot and head sel(U.head, s) + hl (hl > 0 only for packed slots).
template <int D, int MODE>
__device__ __forceinline__ uint16_t* out_row(const TcParams& p, const Unit& U, int s, int tok, int hl) {
    if constexpr (MODE == MODE_PAGED)
        return p.out + ((long)sel(U.qtok, s) + tok) * p.Hq * D + (long)(sel(U.head, s) + hl) * D;
    else
        return p.out + (((long)U.b * p.T + sel(U.row0, s) + tok) * p.Hq + sel(U.head, s)) * D;
}

// A row that sees no key: output 0, LSE -inf (lse may be null).
template <int D>
__device__ __noinline__ void store_zero_row(uint16_t* orow, float* lse) {
    for (int c = 0; c < D; c += 8) *reinterpret_cast<uint4*>(orow + c) = make_uint4(0, 0, 0, 0);
    if (lse) *lse = -INFINITY;
}

// Zeroes rows [z0, z1) of a staged K/V tile (both 64-channel atoms; every
// 16-byte chunk of a row, so the swizzle does not matter) and makes the writes
// visible to the tensor core.  Called by a whole warp.  Kept out of line: the
// call is rare (the last, partly filled block of a context), and inlined into
// the MMA issue loop it slowed that loop by about 10 %.
template <int D>
__device__ __noinline__ void zero_tile_rows(uint8_t* base, int z0, int z1) {
    using C = TcCfg<D>;
    const int n16 = (z1 - z0) * C::kAtoms * 8;
    for (int e = threadIdx.x & 31; e < n16; e += 32) {
        const int row = z0 + e / (C::kAtoms * 8);
        const int a = (e / 8) % C::kAtoms;
        *reinterpret_cast<uint4*>(base + (row >> 3) * C::kPagedGroup + a * 1024 + (row & 7) * 128 + (e % 8) * 16) =
            make_uint4(0, 0, 0, 0);
    }
    fence_proxy_async_smem();
    __syncwarp();
}

// Multiplies this thread's TMEM row of D fp32 columns at taddr by alpha (the
// in-place rescale of O when the running max has grown).  Out of line: it is
// rare after the first tiles, and inlined into the softmax loop it cost about
// 3 % on short prefills.
template <int D>
__device__ __noinline__ void scale_tmem_row(uint32_t taddr, float alpha) {
    __syncwarp();  // warp-collective TMEM accesses follow
#pragma unroll 1
    for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        tmem_ld32(taddr + c * 32, o);
        tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * alpha);
        tmem_st32(taddr + c * 32, o);
    }
    tmem_wait_st();
}

// Pass 1 of the softmax for a tile with additive mask values (class 2): reads
// this thread's 128-column score row from TMEM at taddr, writes back the
// logits s * scale_log2 + M * log2(e) (-inf at columns >= lim), and returns
// their maximum.  mrow: the row's mask values for this tile (null: none);
// vec_mask: they may be read 16 bytes at a time.  Out of line: general tiles
// are rare, and the inlined code slowed every other tile of the loop (and the
// dense kernel, which compiles the same loop).
__device__ __noinline__ float masked_logits_row(uint32_t taddr, const float* mrow, int lim, float scale_log2,
                                                bool vec_mask) {
    float mxp[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) mxp[i] = -INFINITY;
#pragma unroll 1
    for (int h = 0; h < 2; ++h) {
        uint32_t raw[64];
        __syncwarp();  // the TMEM accesses are warp-collective; the mask loads below may diverge
        tmem_ld32(taddr + h * 64, *reinterpret_cast<uint32_t(*)[32]>(raw));
        tmem_ld32(taddr + h * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(raw + 32));
        tmem_wait_ld();
#pragma unroll
        for (int j4 = 0; j4 < 16; ++j4) {
            float mv[4] = {0.f, 0.f, 0.f, 0.f};
            const int j0 = h * 64 + 4 * j4;
            if (vec_mask && j0 + 3 < lim) {
                const float4 t = __ldg(reinterpret_cast<const float4*>(mrow + j0));
                mv[0] = t.x; mv[1] = t.y; mv[2] = t.z; mv[3] = t.w;
            } else if (mrow) {
#pragma unroll
                for (int e = 0; e < 4; ++e) mv[e] = (j0 + e < lim) ? __ldg(mrow + j0 + e) : 0.f;
            }
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int j = j0 + e;
                const float x = j >= lim ? -INFINITY : fmaf(__uint_as_float(raw[4 * j4 + e]), scale_log2, mv[e] * kLog2e);
                raw[4 * j4 + e] = __float_as_uint(x);
                mxp[(4 * j4 + e) & 7] = fmaxf(mxp[(4 * j4 + e) & 7], x);
            }
        }
        __syncwarp();
        tmem_st32(taddr + h * 64, *reinterpret_cast<uint32_t(*)[32]>(raw));
        tmem_st32(taddr + h * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(raw + 32));
    }
    tmem_wait_st();
    return fmaxf(fmaxf(fmaxf(mxp[0], mxp[1]), fmaxf(mxp[2], mxp[3])), fmaxf(fmaxf(mxp[4], mxp[5]), fmaxf(mxp[6], mxp[7])));
}

// The i-th unit of this CTA as the MMA and softmax warps see it: in paged mode
// the one the producer published in mailbox i % kUnitSlots (false if the wait
// gave up), otherwise the static order.
template <int MODE>
__device__ __forceinline__ bool reader_unit(int i, int& u, const TcSched& sched, int G, int num_units,
                                            uint64_t* ufull, uint64_t* uempty, volatile int* umbox,
                                            unsigned long long lim_ns, volatile int* abort_flag) {
    if constexpr (MODE == MODE_PAGED) {
        const int k = i % kUnitSlots;
        if (!mbar_wait_warp(&ufull[k], (i / kUnitSlots) & 1, lim_ns, abort_flag)) return false;
        int v = 0;
        if ((threadIdx.x & 31) == 0) {
            v = umbox[k];
            mbar_arrive(&uempty[k]);
        }
        u = __shfl_sync(0xffffffffu, v, 0);
    } else {
        u = cta_unit(sched, i, G, num_units);
    }
    return true;
}

// Warp-uniform bounded wait that sleeps between polls (for a role with slack,
// so that it leaves its sub-partition's issue slots to the softmax warps).
__device__ __forceinline__ bool mbar_wait_warp_sleepy(uint64_t* bar, uint32_t parity, unsigned long long limit_ns,
                                                      volatile int* abort) {
    bool done = mbar_try_wait(bar, parity);
    if (!done) {
        const uint64_t t0 = globaltimer_ns();
        while (!done) {
            if (*abort || globaltimer_ns() - t0 > limit_ns) break;
            __nanosleep(100);
            done = mbar_try_wait(bar, parity);
        }
    }
    return __all_sync(0xffffffffu, done);
}

// ------------------------------------------------------------------ kernel --
template <int D, int MODE>
__global__ void __launch_bounds__(kTcThreads, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const TcParams p,
                   const __grid_constant__ TcSched sched) {
    using C = TcCfg<D>;
    constexpr int S = C::kStages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    uint8_t* qbuf = smem;
    uint8_t* ring = smem + C::kQBytes;
    uint64_t* full = reinterpret_cast<uint64_t*>(ring + C::kRingBytes);
    uint64_t* empty = full + S;
    uint64_t* qfull = empty + S;
    uint64_t* qempty = qfull + 2;
    uint64_t* sfull = qempty + 2;
    uint64_t* pfull = sfull + 2;  // [slot * 2 + half]: P columns of that half written (and O rescaled);
                                  // the MMA warp waits on half 1, signalled after half 0
    uint64_t* ofull = pfull + 4;
    uint64_t* drain = ofull + 2;
    uint64_t* never = drain + 1;  // nothing arrives on it (forced time-out test hook)
    uint64_t* ufull = never + 1;            // [kUnitSlots] paged mode: unit published in the mailbox
    uint64_t* uempty = ufull + kUnitSlots;  // [kUnitSlots] read by every reader
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(uempty + kUnitSlots);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    volatile int* umbox = abort_flag + 1;  // [kUnitSlots]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int i = 0; i < S; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(&qempty[s], 1);
            mbar_init(&sfull[s], 1);
            mbar_init(&pfull[2 * s], kTcRows);
            mbar_init(&pfull[2 * s + 1], kTcRows);
            mbar_init(&ofull[s], 1);
        }
        mbar_init(drain, 1);
        mbar_init(never, 1);
        *abort_flag = 0;
        mbar_fence_init();
    }
    // The producer's first lane owns the Q barriers' set-up and requests the
    // first unit's Q tiles before the set-up barrier, so that their copies
    // overlap the TMEM allocation and the barrier itself.
    if (warp == kProducerWarp && lane == 0) {
        mbar_init(&qfull[0], 1);
        mbar_init(&qfull[1], 1);
        for (int k = 0; k < kUnitSlots; ++k) {
            mbar_init(&ufull[k], 1);
            mbar_init(&uempty[k], kUnitReaders);
        }
        mbar_fence_init();
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
        int n0;
        if constexpr (MODE == MODE_PAGED)
            n0 = __ldg(p.work_count) * paged_units_per_entry(p);
        else
            n0 = p.num_units;
        const int u0 = cta_unit(sched, 0, gridDim.x, n0);
        if constexpr (MODE == MODE_PAGED) {  // the first unit is this CTA's own: published at once
            umbox[0] = u0;
            mbar_arrive(&ufull[0]);
        }
        if (u0 >= 0) {
            const Unit U0 = decode_unit<MODE>(p, u0);
            if (unit_active<MODE>(p, U0))
                for (int s = 0; s < 2; ++s) {
                    mbar_arrive_expect_tx(&qfull[s], C::kTileBytes);
#pragma unroll
                    for (int a = 0; a < C::kAtoms; ++a) {
                        if constexpr (MODE == MODE_PAGED)
                            tma_load_4d(qbuf + s * C::kTileBytes + a * C::kAtomBytes, &tm_q, &qfull[s], a * 64,
                                        sel(U0.head, s), sel(U0.qtok, s), 0);
                        else
                            tma_load_4d(qbuf + s * C::kTileBytes + a * C::kAtomBytes, &tm_q, &qfull[s], a * 64,
                                        sel(U0.head, s), sel(U0.qtok, s), U0.b);
                    }
                }
        }
    }
    if (warp == kMmaWarp) {
        tmem_alloc(tmem_slot, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *tmem_slot;

    int num_units;
    if constexpr (MODE == MODE_PAGED)
        num_units = __ldg(p.work_count) * paged_units_per_entry(p);
    else
        num_units = p.num_units;
    const int G = gridDim.x;
    const unsigned long long lim_ns = p.ctx.wait_ns;

    auto fail = [&]() {
        raise_error(p.ctx, ERR_TIMEOUT_BIT);
        *abort_flag = 1;
    };

    if (warp == kProducerWarp) {
        // ================================================== TMA producer ====
        int fill = 0, qcnt = 0;
        bool ok = !p.ctx.force_timeout || mbar_wait_warp(never, 0, lim_ns, abort_flag);
        // At kernel start every CTA requests its first Q tiles and its first
        // K/V tiles at once; the rest of the ring waits until the Q tiles are
        // in, so that the first Q K^T is not queued behind the whole ring's
        // copies of every CTA.
        bool held = true;
        for (int i = 0; ok; ++i) {
            int u;
            if constexpr (MODE == MODE_PAGED) {
                // after its first unit a CTA takes the next unit in the longest-first
                // order that no CTA has taken yet, and hands it to the other warps
                u = cta_unit(sched, 0, G, num_units);
                if (i > 0) {
                    int v = -1;
                    if (lane == 0) {
                        const int t = atomicAdd(const_cast<int32_t*>(p.work_count) + 1, 1);
                        v = t < num_units - G ? G + t : -1;
                    }
                    u = __shfl_sync(0xffffffffu, v, 0);
                    const int k = i % kUnitSlots;
                    if (i >= kUnitSlots &&
                        !mbar_wait_warp(&uempty[k], ((i / kUnitSlots) - 1) & 1, lim_ns, abort_flag)) {
                        ok = false;
                        break;
                    }
                    if (lane == 0) {
                        umbox[k] = u;
                        mbar_arrive(&ufull[k]);
                    }
                    __syncwarp();
                }
            } else {
                u = cta_unit(sched, i, G, num_units);
            }
            if (u < 0) break;
            const Unit U = decode_unit<MODE>(p, u);
            if (!unit_active<MODE>(p, U)) continue;
            for (int s = 0; s < 2 && ok && i > 0; ++s) {  // unit 0's Q tiles were requested at the start
                if (!mbar_wait_warp_sleepy(&qempty[s], (qcnt & 1) ^ 1, lim_ns, abort_flag)) {
                    ok = false;
                    break;
                }
                if (lane == 0) {
                    mbar_arrive_expect_tx(&qfull[s], C::kTileBytes);
#pragma unroll
                    for (int a = 0; a < C::kAtoms; ++a) {
                        if constexpr (MODE == MODE_PAGED)
                            tma_load_4d(qbuf + s * C::kTileBytes + a * C::kAtomBytes, &tm_q, &qfull[s], a * 64,
                                        sel(U.head, s), sel(U.qtok, s), 0);
                        else
                            tma_load_4d(qbuf + s * C::kTileBytes + a * C::kAtomBytes, &tm_q, &qfull[s], a * 64,
                                        sel(U.head, s), sel(U.qtok, s), U.b);
                    }
                }
            }
            if (!ok) break;
            ++qcnt;
            // paged: lane j < 8 copies the tile's j-th 16-token block (both
            // 64-channel halves at d = 128); the block-table entries of the next
            // tile are read a tile ahead, so their load latency is off the copy path
            auto load_blk = [&](int kt) -> int {
                const int lb = kt * 8 + lane;
                return (lane < 8 && lb * 16 < U.kv_len) ? __ldg(p.bt + (long)U.b * p.mbps + lb) : 0;
            };
            int blk_next = 0;
            if constexpr (MODE == MODE_PAGED) blk_next = load_blk(U.kt0);
            for (int kt = U.kt0; kt < U.n_kt && ok; ++kt) {
                if (skip_tile<MODE>(p, U, kt)) continue;
                int blk = p.num_blocks;  // outside the map: the copy fills zeros
                if constexpr (MODE == MODE_PAGED) {
                    const int cur = blk_next;
                    if (kt + 1 < U.n_kt) blk_next = load_blk(kt + 1);
                    if (lane < 8 && (kt * 8 + lane) * 16 < U.kv_len) {
                        if (cur < 0 || cur >= p.num_blocks)
                            raise_error(p.ctx, ERR_BOUNDS_BIT);
                        else
                            blk = cur;
                    }
                }
                if (held && fill == 2) {  // first K/V pair issued: let this unit's Q tiles land
                    held = false;
                    for (int s2 = 0; s2 < 2 && ok; ++s2)
                        if (!mbar_wait_warp(&qfull[s2], (qcnt - 1) & 1, lim_ns, abort_flag)) ok = false;
                    if (!ok) break;
                }
                for (int which = 0; which < 2; ++which) {  // 0: K tile, 1: V tile
                    const int stage = fill % S;
                    if (!mbar_wait_warp_sleepy(&empty[stage], ((fill / S) & 1) ^ 1, lim_ns, abort_flag)) {
                        ok = false;
                        break;
                    }
                    uint8_t* dst = ring + stage * C::kTileBytes;
                    const CUtensorMap* tm = which ? &tm_v : &tm_k;
                    if (lane == 0) mbar_arrive_expect_tx(&full[stage], C::kTileBytes);
                    __syncwarp();
                    if constexpr (MODE == MODE_PAGED) {
                        // lane j < 8 copies the tile's j-th 16-token block
                        if (lane < 8) {
                            if constexpr (D == 128)
                                tma_load_5d(dst + lane * 4096, tm, &full[stage], 0, 0, 0, 0, blk * p.Hkv + U.hk);
                            else
                                tma_load_4d(dst + lane * 2048, tm, &full[stage], 0, 0, U.hk, blk);
                        }
                    } else {
                        if (lane == 0) {
#pragma unroll
                            for (int a = 0; a < C::kAtoms; ++a)
                                tma_load_4d(dst + a * C::kAtomBytes, tm, &full[stage], a * 64, U.hk, kt * kTcRows,
                                            U.b);
                        }
                    }
                    __syncwarp();
                    ++fill;
                }
            }
        }
        if (!ok) {
            if (lane == 0) fail();
            // let every copy already issued land before the CTA can exit
            for (int f = max(0, fill - S); f < fill; ++f)
                (void)mbar_wait_warp(&full[f % S], (f / S) & 1, 1000000000ull, nullptr);
            // unit 0's Q tiles may be in flight even if the loop never ran
            bool q0 = false;
            if (qcnt == 0) {
                const int u0 = cta_unit(sched, 0, G, num_units);
                q0 = u0 >= 0 && unit_active<MODE>(p, decode_unit<MODE>(p, u0));
            }
            if (qcnt > 0 || q0)
                for (int s = 0; s < 2; ++s)
                    (void)mbar_wait_warp(&qfull[s], qcnt > 0 ? (qcnt - 1) & 1 : 0, 1000000000ull, nullptr);
        }
    } else if (warp == kMmaWarp) {
        // ===================================================== MMA issuer ===
        constexpr uint32_t kIdescQK = idesc_bf16_f32(128, 128, 0, 0);
        constexpr uint32_t kIdescPV = idesc_bf16_f32(128, D, 0, 1);
        const uint32_t q_addr = smem_u32(qbuf), ring_addr = smem_u32(ring);
        auto s_col = [](int s) -> uint32_t { return s ? C::kS1 : C::kS0; };
        auto o_col = [](int s) -> uint32_t { return s ? C::kO1 : C::kO0; };
        int cons = 0, ucnt = 0, pc0 = 0, pc1 = 0;  // pc: P tiles consumed per slot
        bool ok = !p.ctx.force_timeout || mbar_wait_warp(never, 0, lim_ns, abort_flag);

        // `ready`: the phase was already seen complete by every lane (mbar_test3)
        auto wait_v = [&](int vidx, int vkt, int kv_len, bool ready = false) -> bool {
            if (!ready && !mbar_wait_warp(&full[vidx % S], (vidx / S) & 1, lim_ns, abort_flag)) return false;
            if constexpr (MODE == MODE_PAGED) {
                // Rows past the context inside the last partly filled block
                // may hold stale words; zero them so a zero probability never
                // meets a non-finite value.
                const int kv0 = vkt * kTcRows;
                const int z0 = kv_len - kv0;
                const int z1 = min(kTcRows, ((kv_len + 15) & ~15) - kv0);
                if (z0 < z1) zero_tile_rows<D>(ring + (vidx % S) * C::kTileBytes, z0, z1);
            }
            return true;
        };
        // The start-address field of a descriptor is (address >> 4) in 14 bits;
        // shared addresses stay below 256 KB, so advancing a descriptor by a byte
        // offset is adding offset >> 4.
        // K/V tile layout: 8-row groups kv_sbo bytes apart, 64-channel halves kv_half apart
        constexpr uint32_t kv_sbo = MODE == MODE_PAGED ? C::kPagedGroup : 1024;
        constexpr uint32_t kv_half = MODE == MODE_PAGED ? 1024 : C::kAtomBytes;
        auto issue_qk = [&](int s, int kidx) {
            const uint64_t kd = smem_desc_sw128(ring_addr + (kidx % S) * C::kTileBytes, 16, kv_sbo);
            const uint64_t qd = smem_desc_sw128(q_addr + s * C::kTileBytes, 16, 1024);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const uint32_t qoff = ((kk >> 2) * C::kAtomBytes + (kk & 3) * 32) >> 4;
                const uint32_t koff = ((kk >> 2) * kv_half + (kk & 3) * 32) >> 4;
                umma_ss(tbase + s_col(s), qd + qoff, kd + koff, kIdescQK, kk > 0);
            }
        };
        // O_s += P_s V over keys [64h, 64h+64) of the tile
        auto issue_pv_half = [&](int s, int vidx, int h, bool acc_first) {
            const uint64_t vd = smem_desc_sw128(ring_addr + (vidx % S) * C::kTileBytes, kv_half, kv_sbo);
#pragma unroll
            for (int k4 = 0; k4 < 4; ++k4) {
                const int kk = 4 * h + k4;  // keys [16 kk, 16 kk + 16): two 8-row groups
                umma_ts(tbase + o_col(s), tbase + s_col(s) + kk * 8, vd + (uint32_t)(kk * 2 * kv_sbo >> 4), kIdescPV,
                        (acc_first || kk > 0));
            }
        };
        // waits for P_s and issues its P*V MMAs.  The second half is signalled
        // after the first, so one wait covers both.
        auto pv = [&](int s, int vidx, bool acc_first, bool ready = false) -> bool {
            if (!ready && !mbar_wait_warp(&pfull[2 * s + 1], (s ? pc1 : pc0) & 1, lim_ns, abort_flag)) return false;
            tc_fence_after();
            if (lane == 0) {
                issue_pv_half(s, vidx, 0, acc_first);
                issue_pv_half(s, vidx, 1, acc_first);
            }
            __syncwarp();
            if (s) ++pc1;
            else ++pc0;
            return true;
        };

        for (int i = 0; ok; ++i) {
            int u;
            if (!reader_unit<MODE>(i, u, sched, G, num_units, ufull, uempty, umbox, lim_ns, abort_flag)) {
                ok = false;
                break;
            }
            if (u < 0) break;
            const Unit U = decode_unit<MODE>(p, u);
            if (!unit_active<MODE>(p, U)) continue;
            // the next unit's Q tiles take ~1 us to land: a sleeping wait leaves the
            // sub-partition's issue slots to the softmax warps' epilogue
            for (int s = 0; s < 2; ++s)
                if (!mbar_wait_warp_sleepy(&qfull[s], ucnt & 1, lim_ns, abort_flag)) ok = false;
            if (!ok) break;
            ++ucnt;
            int it = 0, prev_v = -1, prev_kt = -1;
            for (int kt = U.kt0; kt < U.n_kt && ok; ++kt) {
                if (skip_tile<MODE>(p, U, kt)) continue;
                const int kidx = cons + 2 * it;
                // Before slot 0's MMAs the previous V tile, P_0 and this K tile are
                // probed together: each barrier check in this warp costs the tensor
                // pipe idle time, and three probes in flight cost about one.
                // (Paged K tiles arrive box by box and are rarely complete this
                // early, so paged mode waits as before.)
                bool v_rdy = false, p0_rdy = false, k_rdy = false;
                if (MODE != MODE_PAGED && it > 0) {
                    uint32_t r[3];
                    mbar_test3(&full[prev_v % S], (prev_v / S) & 1, &pfull[1], pc0 & 1, &full[kidx % S],
                               (kidx / S) & 1, r);
                    v_rdy = __all_sync(0xffffffffu, r[0]);
                    p0_rdy = __all_sync(0xffffffffu, r[1]);
                    k_rdy = __all_sync(0xffffffffu, r[2]);
                }
                for (int s = 0; s < 2 && ok; ++s) {
                    // P_s V of the previous tile goes out as soon as P_s is
                    // ready; only the Q K^T after it waits for this tile's K
                    if (it > 0) {
                        if (s == 0 && !wait_v(prev_v, prev_kt, U.kv_len, v_rdy)) {
                            ok = false;
                            break;
                        }
                        if (!pv(s, prev_v, it > 1, s == 0 && p0_rdy)) {
                            ok = false;
                            break;
                        }
                    }
                    if (s == 0) {
                        if (!k_rdy && !mbar_wait_warp(&full[kidx % S], (kidx / S) & 1, lim_ns, abort_flag)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                    }
                    if (lane == 0) {
                        issue_qk(s, kidx);
                        umma_commit(&sfull[s]);
                    }
                    __syncwarp();
                }
                if (!ok) break;
                if (lane == 0) {
                    umma_commit(&empty[kidx % S]);
                    if (it > 0) umma_commit(&empty[prev_v % S]);
                }
                __syncwarp();
                prev_v = kidx + 1;
                prev_kt = kt;
                ++it;
            }
            if (!ok) break;
            if (lane == 0) {
                umma_commit(&qempty[0]);
                umma_commit(&qempty[1]);
            }
            if (!wait_v(prev_v, prev_kt, U.kv_len)) {
                ok = false;
                break;
            }
            for (int s = 0; s < 2 && ok; ++s) {
                if (!pv(s, prev_v, it > 1)) {
                    ok = false;
                    break;
                }
                if (lane == 0) umma_commit(&ofull[s]);
                __syncwarp();
            }
            if (!ok) break;
            if (lane == 0) umma_commit(&empty[prev_v % S]);
            __syncwarp();
            cons += 2 * it;
        }
        if (!ok && lane == 0) fail();
        // every MMA issued above completes before TMEM is released
        if (lane == 0) umma_commit(drain);
        __syncwarp();
        (void)mbar_wait_bounded(drain, 0, 1000000000ull, nullptr);
    } else {
        // ======================================================== softmax ===
        const int s = warp >> 2;
        const int quarter = warp & 3;
        const int r = quarter * 32 + lane;
        const uint32_t trow = tbase + ((uint32_t)(quarter * 32) << 16);
        const uint32_t s_col = s ? C::kS1 : C::kS0;
        const uint32_t o_col = s ? C::kO1 : C::kO0;
        int sc = 0, oc = 0;
        bool ok = !p.ctx.force_timeout || mbar_wait_warp(never, 0, lim_ns, abort_flag);
        for (int i = 0; ok; ++i) {
            int u;
            if (!reader_unit<MODE>(i, u, sched, G, num_units, ufull, uempty, umbox, lim_ns, abort_flag)) {
                ok = false;
                break;
            }
            if (u < 0) break;
            const Unit U = decode_unit<MODE>(p, u);
            // query token of this thread's row, and its head within a packed slot
            const int tok = (MODE == MODE_PAGED && p.pack) ? r >> p.pack_shift : r;
            const int hl = (MODE == MODE_PAGED && p.pack) ? r & (p.g - 1) : 0;
            const bool valid = tok < sel(U.nrows, s);
            const int row = sel(U.row0, s) + tok;  // row within T (dense) or within the chunk (paged)
            if (!unit_active<MODE>(p, U)) {
                if (valid) {
                    float* lse = nullptr;
                    if constexpr (MODE != MODE_PAGED)
                        if (p.lse) lse = p.lse + ((long)U.b * p.Hq + sel(U.head, s)) * p.T + row;
                    store_zero_row<D>(out_row<D, MODE>(p, U, s, tok, hl), lse);
                }
                continue;
            }
            // key j is visible when j <= row + pos_off (causal) and j < kv_len
            const int vis_end = p.causal ? min(U.kv_len, row + U.pos_off + 1) : U.kv_len;
            float m = -INFINITY, l = 0.f;
            int it = 0;
            // masked mode: this slot's class of the next tile and, for a class-3
            // tile, this row's run of keys, read a tile ahead (a unit without
            // holes visits every tile of its range)
            const int nkt = (p.T + kTcRows - 1) / kTcRows;
            auto row_run = [&](int kt) -> uchar2 {
                return __ldg(reinterpret_cast<const uchar2*>(p.iv) +
                             ((long)(sel(U.row0, s) / kTcRows) * nkt + kt) * kTcRows + r);
            };
            int cls_next = 0;
            uchar2 run_next = make_uchar2(0, 0);
            if constexpr (MODE == MODE_MASKED) {
                cls_next = tile_class<MODE>(p, U, s, U.kt0);
                if (cls_next == 3) run_next = row_run(U.kt0);
            }
            for (int kt = U.kt0; kt < U.n_kt; ++kt) {
                if (skip_tile<MODE>(p, U, kt)) continue;
                int cls;
                uchar2 run = make_uchar2(0, 0);
                if constexpr (MODE == MODE_MASKED) {
                    if (U.holes) {
                        cls = tile_class<MODE>(p, U, s, kt);
                        if (cls == 3) run = row_run(kt);
                    } else {
                        cls = cls_next;
                        run = run_next;
                        if (kt + 1 < U.n_kt) {
                            cls_next = tile_class<MODE>(p, U, s, kt + 1);
                            if (cls_next == 3) run_next = row_run(kt + 1);
                        }
                    }
                } else {
                    cls = tile_class<MODE>(p, U, s, kt);
                }
                if (!mbar_wait_warp(&sfull[s], sc & 1, lim_ns, abort_flag)) {
                    ok = false;
                    break;
                }
                ++sc;
                tc_fence_after();
                const int kv0 = kt * kTcRows;
                const int lim = vis_end - kv0;  // visible columns of this tile: [0, lim)
                const float* mrow = (cls == 2 && valid) ? p.mask + (long)row * p.T + kv0 : nullptr;
                // cls is the same for the whole warp (it depends on the slot and the
                // tile only).  Without mask values (cls 0 or 1) the scores need only
                // the scale and the column limit, both applied in registers; with
                // mask values (cls 2, "general") the masked, scaled logits are
                // written back over S in pass 1 so that pass 2 reads them instead of
                // re-reading the mask.
                const bool general = cls == 2;
                // visible columns of this row: [vlo, vlim); a class-3 tile keeps
                // the row's run of keys, applied like the causal limit (the
                // limit path takes the general path's operations, so both give
                // the same bits)
                int vlo = 0, vlim = cls == 0 ? 0 : lim;
                if constexpr (MODE == MODE_MASKED)
                    if (cls == 3) {
                        vlo = run.x;
                        vlim = min(lim, (int)run.y);
                    }
                // every column of every row of the warp visible and no mask values
                const bool plain = !general && __all_sync(0xffffffffu, vlo == 0 && vlim >= kTcRows);
                // pass 1: row max.  Without mask values the whole 128-column score row
                // is loaded with one TMEM wait; the general case takes 64 columns per
                // wait.  8 independent partial maxima / sums keep the reductions off a
                // single serial dependency chain.
                float mxp[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) mxp[i] = -INFINITY;
                if (!general) {  // scale > 0: the max of the raw scores gives the max of the scaled ones
                    uint32_t raw[kTcRows];
#pragma unroll
                    for (int c = 0; c < kTcRows / 32; ++c)
                        tmem_ld32(trow + s_col + c * 32, *reinterpret_cast<uint32_t(*)[32]>(raw + 32 * c));
                    tmem_wait_ld();
                    if (plain) {
#pragma unroll
                        for (int j = 0; j < kTcRows; j += 2)
                            mxp[(j >> 1) & 7] =
                                fmax3f(mxp[(j >> 1) & 7], __uint_as_float(raw[j]), __uint_as_float(raw[j + 1]));
                    } else {
#pragma unroll
                        for (int j = 0; j < kTcRows; j += 2)
                            mxp[(j >> 1) & 7] =
                                fmax3f(mxp[(j >> 1) & 7], j >= vlo && j < vlim ? __uint_as_float(raw[j]) : -INFINITY,
                                       j + 1 >= vlo && j + 1 < vlim ? __uint_as_float(raw[j + 1]) : -INFINITY);
                    }
                } else {
                    mxp[0] = masked_logits_row(trow + s_col, mrow, lim, p.scale_log2, mrow && ((p.T & 3) == 0));
                }
                float mx = fmaxf(fmaxf(fmaxf(mxp[0], mxp[1]), fmaxf(mxp[2], mxp[3])),
                                 fmaxf(fmaxf(mxp[4], mxp[5]), fmaxf(mxp[6], mxp[7])));
                if (!general) mx *= p.scale_log2;
                const float m_new = fmaxf(m, mx);
                const bool need = m_new > m + kRescaleThreshold;
                float alpha = 1.f;
                const bool warp_rescale = __any_sync(0xffffffffu, need);
                if (warp_rescale) {
                    alpha = (m == -INFINITY) ? 0.f : fast_exp2(m - m_new);
                    l *= alpha;
                    m = m_new;
                }
                const float m_use = (m == -INFINITY) ? 0.f : m;
                // O must be rescaled before the first P*V of this tile: in that
                // (rare) case both halves are signalled after the rescale
                const bool rescale_o = warp_rescale && it > 0;
                // pass 2: P = 2^(logit - m) as bf16.  Half h reads S columns
                // [64h, 64h+64) and writes P columns [32h, 32h+32), only over S
                // columns already read.  Without a rescale each half is signalled as
                // soon as it is stored; the MMA warp waits on the second half only
                // (one barrier check instead of two), but signalling the first
                // half early, with its store wait, measured faster than one
                // signal at the end.  Column pairs go through packed f32x2 FMA /
                // add (one instruction per pair).
                float2 rsp[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                                 make_float2(0.f, 0.f)};
                const float sc = general ? 1.f : p.scale_log2;  // logits already scaled in the general case
                const float2 sc2 = make_float2(sc, sc), neg_m = make_float2(-m_use, -m_use);
#pragma unroll 1
                for (int h = 0; h < 2; ++h) {
                    uint32_t raw[64];
                    tmem_ld32(trow + s_col + h * 64, *reinterpret_cast<uint32_t(*)[32]>(raw));
                    tmem_ld32(trow + s_col + h * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(raw + 32));
                    tmem_wait_ld();
                    uint32_t pk[32];
                    if (plain || general) {  // every column visible, or masked logits already -inf
#pragma unroll
                        for (int j = 0; j < 32; ++j) {
                            const float2 x = __ffma2_rn(
                                make_float2(__uint_as_float(raw[2 * j]), __uint_as_float(raw[2 * j + 1])), sc2, neg_m);
                            const float2 pp = make_float2(fast_exp2(x.x), fast_exp2(x.y));
                            rsp[j & 3] = __fadd2_rn(rsp[j & 3], pp);
                            pk[j] = pack_bf16x2(pp.x, pp.y);
                        }
                    } else {
                        // columns at or past the row's limit get probability 0.  The
                        // logit takes the general case's operations (scaled with a zero
                        // addend, then the max subtracted), so that a causal limit and
                        // an additive -inf mask of the same shape give bit-identical
                        // results.
                        const int c0 = h * 64;
#pragma unroll
                        for (int j = 0; j < 32; ++j) {
                            const float2 x = __ffma2_rn(make_float2(fmaf(__uint_as_float(raw[2 * j]), p.scale_log2, 0.f),
                                                                    fmaf(__uint_as_float(raw[2 * j + 1]), p.scale_log2, 0.f)),
                                                        make_float2(1.f, 1.f), neg_m);
                            const int cj = c0 + 2 * j;
                            const float2 pp = make_float2(cj >= vlo && cj < vlim ? fast_exp2(x.x) : 0.f,
                                                          cj + 1 >= vlo && cj + 1 < vlim ? fast_exp2(x.y) : 0.f);
                            rsp[j & 3] = __fadd2_rn(rsp[j & 3], pp);
                            pk[j] = pack_bf16x2(pp.x, pp.y);
                        }
                    }
                    tmem_st32(trow + s_col + h * 32, pk);
                    if (!rescale_o) {
                        tmem_wait_st();
                        tc_fence_before();
                        mbar_arrive(&pfull[2 * s + h]);
                    }
                }
                l += ((rsp[0].x + rsp[0].y) + (rsp[1].x + rsp[1].y)) + ((rsp[2].x + rsp[2].y) + (rsp[3].x + rsp[3].y));
                if (rescale_o) {
                    scale_tmem_row<D>(trow + o_col, alpha);
                    tc_fence_before();
                    mbar_arrive(&pfull[2 * s]);
                    mbar_arrive(&pfull[2 * s + 1]);
                }
                ++it;
            }
            if (!ok) break;
            if (!mbar_wait_warp(&ofull[s], oc & 1, lim_ns, abort_flag)) {
                ok = false;
                break;
            }
            ++oc;
            tc_fence_after();
            const Unit E = decode_unit<MODE>(p, u);  // re-derived here so its fields are not live across the tile loop
            uint16_t* orow = out_row<D, MODE>(p, E, s, tok, hl);
            const float inv_l = l > 0.f ? 1.f / l : 0.f;
            // 64 columns per TMEM wait; 32-byte stores of the bf16 row
#pragma unroll
            for (int c = 0; c < D / 64; ++c) {
                uint32_t raw[64];
                tmem_ld32(trow + o_col + c * 64, *reinterpret_cast<uint32_t(*)[32]>(raw));
                tmem_ld32(trow + o_col + c * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(raw + 32));
                tmem_wait_ld();
                uint32_t pk[32];
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    pk[j] = pack_bf16x2(__uint_as_float(raw[2 * j]) * inv_l, __uint_as_float(raw[2 * j + 1]) * inv_l);
                if (valid) {
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4)
                        st_global_v8(orow + c * 64 + q4 * 16, pk[8 * q4], pk[8 * q4 + 1], pk[8 * q4 + 2],
                                     pk[8 * q4 + 3], pk[8 * q4 + 4], pk[8 * q4 + 5], pk[8 * q4 + 6], pk[8 * q4 + 7]);
                }
            }
            if constexpr (MODE != MODE_PAGED)
                if (p.lse && valid)
                    p.lse[((long)E.b * p.Hq + sel(E.head, s)) * p.T + row] = l > 0.f ? (m + __log2f(l)) * kLn2 : -INFINITY;
        }
        if (!ok && lane == 0) fail();
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kMmaWarp) tmem_dealloc(tbase, 512);
}

// ----------------------------------------------------------- mask order ---
// Orders query tiles by decreasing number of KV tiles that are not entirely
// masked (longest first), from the tile classes of the additive mask.
__global__ void __launch_bounds__(256) mask_order_kernel(const uint8_t* __restrict__ cls, int nqt, int nkt,
                                                         int causal, int32_t* __restrict__ order,
                                                         int2* __restrict__ range) {
    extern __shared__ int cost[];
    // one warp per query tile, 32 of its classes per (coalesced) step
    const int lane = threadIdx.x & 31, nw = blockDim.x >> 5;
    for (int q = threadIdx.x >> 5; q < nqt; q += nw) {
        int c = 0, lo = nkt, hi = 0;
        const int kend = causal ? min(nkt, q + 1) : nkt;
        for (int k0 = 0; k0 < kend; k0 += 32) {
            const int k = k0 + lane;
            const unsigned vis = __ballot_sync(0xffffffffu, k < kend && cls[(long)q * nkt + k] != 0);
            if (vis) {
                c += __popc(vis);
                if (lo == nkt) lo = k0 + __ffs(vis) - 1;
                hi = k0 + 32 - __clz(vis);
            }
        }
        if (lane == 0) {
            cost[q] = c;
            // flag: an all -inf tile inside [lo, hi) (the scan must check classes)
            range[q] = make_int2(lo | (c > 0 && c < hi - lo ? kRangeHoles : 0), hi);
        }
    }
    __syncthreads();
    for (int q = threadIdx.x; q < nqt; q += blockDim.x) {
        int rank = 0;
        const int cq = cost[q];
        for (int o = 0; o < nqt; ++o) rank += (cost[o] > cq) || (cost[o] == cq && o < q);
        order[rank] = q;
    }
}

fa_status launch_mask_classify(const float* M, int Tq, int Tk, uint8_t* cls, uint8_t* iv, cudaStream_t s);

// ------------------------------------------------------------ launchers ---
template <int D, int MODE>
static fa_status launch_tc(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const TcParams& p,
                           int grid, cudaStream_t s, const TcSched& sched) {
    const fa_status st = raise_dynamic_smem(reinterpret_cast<const void*>(attn_tc_kernel<D, MODE>), TcCfg<D>::kSmem);
    if (st != FA_OK) return st;
    attn_tc_kernel<D, MODE><<<grid, kTcThreads, TcCfg<D>::kSmem, s>>>(tq, tk, tv, p, sched);
    return cuda_status(cudaGetLastError());
}

template <int MODE>
static fa_status launch_tc_d(int d, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                             const TcParams& p, int grid, cudaStream_t s, const TcSched* sched = nullptr) {
    static const TcSched kNone = {};  // n == 0: the unit_of order
    const TcSched& sc = sched ? *sched : kNone;
    return d == 128 ? launch_tc<128, MODE>(tq, tk, tv, p, grid, s, sc) : launch_tc<64, MODE>(tq, tk, tv, p, grid, s, sc);
}

// Balanced unit-to-CTA assignment for dense causal prefill.  A unit's cost is
// its KV tiles plus a fixed start/epilogue cost of about 1.4 tiles (measured);
// units go longest first to the least loaded CTA, then single moves and swaps
// off the most loaded CTA continue while they lower the maximum (at most 4000
// steps, stopping within 0.5 % of the mean load).
// Cached per (B, T, Hq, Hkv, grid): the result depends on nothing else.
static const TcSched* dense_schedule(const TcParams& p, int grid) {
    if (!p.causal || p.num_units > kMaxSchedUnits || grid > kMaxSchedCtas || grid <= 0) return nullptr;
    if (p.q0 != 0 || p.Tq != p.T || p.Tk != p.T) return nullptr;  // row windows take the dealt order
    struct Key {
        int B, T, Hq, Hkv, grid;
        bool operator==(const Key& o) const {
            return B == o.B && T == o.T && Hq == o.Hq && Hkv == o.Hkv && grid == o.grid;
        }
    };
    static std::mutex mu;
    static std::vector<std::pair<Key, std::unique_ptr<TcSched>>> cache;
    const Key key{p.B, p.T, p.Hq, p.Hkv, grid};
    std::lock_guard<std::mutex> lk(mu);
    for (auto& e : cache)
        if (e.first == key) return e.second.get();
    // unit costs, in the unit numbering decode_unit uses (rank-major, longest first)
    const int nqt = (p.T + kTcRows - 1) / kTcRows, n = p.num_units;
    std::vector<double> cost(n);
    for (int u = 0; u < n; ++u) {
        int kt;
        if (p.pair_heads) {
            const int upt = p.B * p.Hkv * (p.g / 2);
            kt = nqt - u / upt;  // query tile nqt - 1 - rank sees qt + 1 KV tiles
        } else {
            const int upt = p.B * p.Hq, ntp = (nqt + 1) / 2;
            kt = std::min(nqt, 2 * (ntp - 1 - u / upt) + 2);
        }
        cost[u] = kt + 1.4;
    }
    std::vector<std::vector<int>> bins(grid);
    std::vector<double> load(grid, 0.0);
    for (int u = 0; u < n; ++u) {  // u already runs longest first
        const int b = (int)(std::min_element(load.begin(), load.end()) - load.begin());
        bins[b].push_back(u);
        load[b] += cost[u];
    }
    double mean = 0.0;
    for (double x : load) mean += x;
    mean /= grid;
    for (int iter = 0; iter < 4000; ++iter) {
        const int a = (int)(std::max_element(load.begin(), load.end()) - load.begin());
        if (load[a] <= mean * 1.005) break;  // within 0.5 % of the ideal
        bool moved = false;
        for (int b = 0; b < grid && !moved; ++b) {
            if (b == a) continue;
            for (size_t i = 0; i < bins[a].size() && !moved; ++i) {
                const int x = bins[a][i];
                if (load[b] + cost[x] < load[a] - 1e-9) {
                    bins[b].push_back(x);
                    bins[a].erase(bins[a].begin() + i);
                    load[b] += cost[x];
                    load[a] -= cost[x];
                    moved = true;
                    break;
                }
                for (size_t j = 0; j < bins[b].size(); ++j) {
                    const int y = bins[b][j];
                    const double na = load[a] - cost[x] + cost[y], nb = load[b] - cost[y] + cost[x];
                    if (cost[y] < cost[x] && na < load[a] - 1e-9 && nb < load[a] - 1e-9) {
                        bins[a][i] = y;
                        bins[b][j] = x;
                        load[a] = na;
                        load[b] = nb;
                        moved = true;
                        break;
                    }
                }
            }
        }
        if (!moved) break;
    }
    auto sc = std::make_unique<TcSched>();
    sc->n = n;
    int k = 0;
    for (int c = 0; c < grid; ++c) {
        std::sort(bins[c].begin(), bins[c].end());  // longest first within the CTA
        sc->start[c] = (uint16_t)k;
        for (int u : bins[c]) sc->unit[k++] = (uint16_t)u;
    }
    sc->start[grid] = (uint16_t)k;
    cache.emplace_back(key, std::move(sc));
    return cache.back().second.get();
}

static fa_status dense_maps(const void* q, const void* k, const void* v, int B, int T, int Hq, int Hkv, int d,
                            CUtensorMap* tq, CUtensorMap* tk, CUtensorMap* tv) {
    const uint32_t box[4] = {64, 1, (uint32_t)kTcRows, 1};
    const uint64_t dq[4] = {(uint64_t)d, (uint64_t)Hq, (uint64_t)T, (uint64_t)B};
    const uint64_t sq[3] = {(uint64_t)d * 2, (uint64_t)Hq * d * 2, (uint64_t)T * Hq * d * 2};
    const uint64_t dk[4] = {(uint64_t)d, (uint64_t)Hkv, (uint64_t)T, (uint64_t)B};
    const uint64_t sk[3] = {(uint64_t)d * 2, (uint64_t)Hkv * d * 2, (uint64_t)T * Hkv * d * 2};
    fa_status st = encode_tmap_bf16_4d(tq, q, dq, sq, box);
    if (st == FA_OK) st = encode_tmap_bf16_4d(tk, k, dk, sk, box);
    if (st == FA_OK) st = encode_tmap_bf16_4d(tv, v, dk, sk, box);
    return st;
}

static fa_status check_prefill_args(const void* q, const void* k, const void* v, const void* out, int B, int T,
                                    int Hq, int Hkv, int d, float scale) {
    if (B < 0 || T < 0 || Hq <= 0 || Hkv <= 0 || !(scale > 0.f) || !std::isfinite(scale)) return FA_ERR_INVALID_ARG;
    if ((d != 64 && d != 128) || Hq % Hkv != 0) return FA_ERR_UNSUPPORTED;
    if (B == 0 || T == 0) return FA_OK;
    if (!q || !k || !v || !out) return FA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned32(out)) return FA_ERR_INVALID_ARG;
    return FA_OK;
}

static TcParams base_params(int B, int T, int Hq, int Hkv, int causal, float scale, void* out, float* lse,
                            const DevCtx& ctx) {
    TcParams p{};
    p.B = B;
    p.T = T;
    p.q0 = 0;
    p.Tq = T;
    p.Tk = T;
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.g = Hq / Hkv;
    p.causal = causal ? 1 : 0;
    p.scale_log2 = scale * kLog2e;
    p.pair_heads = (p.g % 2 == 0) ? 1 : 0;
    p.out = static_cast<uint16_t*>(out);
    p.lse = lse;
    p.ctx = ctx;
    return p;
}

static int dense_units(const TcParams& p) {
    const int nqt = (p.Tq + kTcRows - 1) / kTcRows;
    return p.pair_heads ? p.B * p.Hkv * (p.g / 2) * nqt : p.B * p.Hq * ((nqt + 1) / 2);
}

fa_status launch_paged_prefill(const void* q, const void* k_cache, const void* v_cache, const int32_t* block_table,
                               const int32_t* ctx_lens, const int32_t* q_lens, const int32_t* q_start,
                               const int32_t* work_list, const int32_t* work_count, void* out, int num_seqs,
                               int mbps, int num_blocks, int Hq, int Hkv, int d, int causal, float scale,
                               int total_q, cudaStream_t s, const DevCtx& ctx) {
    (void)num_seqs;
    CUtensorMap tq, tk, tv;
    const int g = Hq / Hkv;
    const bool pack = paged_tc_pack(g);
    // packed: one box is 128/g tokens x the g heads of a group (row = token * g + head)
    const uint32_t qbox[4] = {64, pack ? (uint32_t)g : 1u, (uint32_t)paged_tc_slot_tokens(g), 1};
    const uint64_t dq[4] = {(uint64_t)d, (uint64_t)Hq, (uint64_t)total_q, 1};
    const uint64_t sq[3] = {(uint64_t)d * 2, (uint64_t)Hq * d * 2, (uint64_t)total_q * Hq * d * 2};
    fa_status st = encode_tmap_bf16_4d(&tq, q, dq, sq, qbox);
    if (d == 128) {
        // one box per (block, kv head): 64 channels x 8 rows x 2 halves x 2 row groups,
        // landing as [group][half][8 rows][128 B]; the last dimension is block * Hkv + head
        const uint32_t cbox[5] = {64, 8, 2, 2, 1};
        const uint64_t dc[5] = {64, 8, 2, 2, (uint64_t)num_blocks * Hkv};
        const uint64_t scs[4] = {256, 128, 2048, 4096};
        if (st == FA_OK) st = encode_tmap_bf16_5d(&tk, k_cache, dc, scs, cbox);
        if (st == FA_OK) st = encode_tmap_bf16_5d(&tv, v_cache, dc, scs, cbox);
    } else {
        const uint32_t cbox[4] = {64, 16, 1, 1};
        const uint64_t dc[4] = {(uint64_t)d, 16, (uint64_t)Hkv, (uint64_t)num_blocks};
        const uint64_t scs[3] = {(uint64_t)d * 2, (uint64_t)16 * d * 2, (uint64_t)Hkv * 16 * d * 2};
        if (st == FA_OK) st = encode_tmap_bf16_4d(&tk, k_cache, dc, scs, cbox);
        if (st == FA_OK) st = encode_tmap_bf16_4d(&tv, v_cache, dc, scs, cbox);
    }
    if (st != FA_OK) return st;
    TcParams p = base_params(0, 0, Hq, Hkv, causal, scale, out, nullptr, ctx);
    p.pack = pack ? 1 : 0;
    p.pack_shift = pack ? __builtin_ctz((unsigned)g) : 0;
    p.bt = block_table;
    p.ctx_lens = ctx_lens;
    p.q_lens = q_lens;
    p.q_start = q_start;
    p.work_list = work_list;
    p.work_count = work_count;
    p.mbps = mbps;
    p.num_blocks = num_blocks;
    return launch_tc_d<MODE_PAGED>(d, tq, tk, tv, p, sm_count(), s);
}

// Query rows [q0, q0 + Tq) of every sequence against keys [0, Tk), for the
// host pipeline: arguments as fa_prefill's (already checked by the caller),
// q0 a multiple of 128, q0 + Tq <= T, Tk <= T.  The rows computed here are bit
// for bit those of the whole-problem call: the same query tiles meet the same
// key tiles in the same order.
fa_status launch_prefill_rows(const void* q, const void* k, const void* v, void* out, int B, int T, int Hq, int Hkv,
                              int d, int causal, float scale, int q0, int Tq, int Tk, cudaStream_t s) {
    if (q0 < 0 || (q0 % kTcRows) != 0 || Tq <= 0 || q0 + Tq > T || Tk <= 0 || Tk > T) return FA_ERR_INVALID_ARG;
    DevCtx ctx;
    fa_status st = make_ctx(&ctx);
    if (st != FA_OK) return st;
    CUtensorMap tq, tk, tv;
    if ((st = dense_maps(q, k, v, B, T, Hq, Hkv, d, &tq, &tk, &tv)) != FA_OK) return st;
    TcParams p = base_params(B, T, Hq, Hkv, causal, scale, out, nullptr, ctx);
    p.q0 = q0;
    p.Tq = Tq;
    p.Tk = Tk;
    p.num_units = dense_units(p);
    const int grid = std::min(p.num_units, sm_count());
    return launch_tc_d<MODE_DENSE>(d, tq, tk, tv, p, grid, s, dense_schedule(p, grid));
}

}  // namespace fa

using namespace fa;

extern "C" {

fa_status fa_prefill(const void* q, const void* k, const void* v, void* out, int B, int T, int Hq, int Hkv, int d,
                     int causal, float scale, float* lse, fa_stream_t stream) {
    set_launch_count(0);
    fa_status st = check_prefill_args(q, k, v, out, B, T, Hq, Hkv, d, scale);
    if (st != FA_OK || B == 0 || T == 0) return st;
    if ((st = check_device()) != FA_OK) return st;
    DevCtx ctx;
    if ((st = make_ctx(&ctx)) != FA_OK) return st;
    CUtensorMap tq, tk, tv;
    if ((st = dense_maps(q, k, v, B, T, Hq, Hkv, d, &tq, &tk, &tv)) != FA_OK) return st;
    TcParams p = base_params(B, T, Hq, Hkv, causal, scale, out, lse, ctx);
    p.num_units = dense_units(p);
    const int grid = std::min(p.num_units, sm_count());
    st = launch_tc_d<MODE_DENSE>(d, tq, tk, tv, p, grid, reinterpret_cast<cudaStream_t>(stream),
                                 dense_schedule(p, grid));
    if (st == FA_OK) set_launch_count(1);
    return st;
}

fa_status fa_prefill_rows(const void* q, const void* k, const void* v, void* out, int B, int T, int Hq, int Hkv,
                          int d, int causal, float scale, int q0, int Tq, int Tk, fa_stream_t stream) {
    set_launch_count(0);
    fa_status st = check_prefill_args(q, k, v, out, B, T, Hq, Hkv, d, scale);
    if (st != FA_OK || B == 0 || T == 0 || Tq == 0) return st;
    if (q0 < 0 || (q0 % kTcRows) != 0 || Tq < 0 || q0 + Tq > T || Tk <= 0 || Tk > T || (causal && Tk < q0 + Tq))
        return FA_ERR_INVALID_ARG;
    if ((st = check_device()) != FA_OK) return st;
    st = launch_prefill_rows(q, k, v, out, B, T, Hq, Hkv, d, causal, scale, q0, Tq, Tk,
                             reinterpret_cast<cudaStream_t>(stream));
    if (st == FA_OK) set_launch_count(1);
    return st;
}

size_t fa_prefill_masked_workspace_size(int T) {
    if (T <= 0) return 0;
    const size_t nt = (size_t)(T + kTcRows - 1) / kTcRows;
    return align256(nt * nt) + align256(sizeof(int32_t) * nt) + align256(sizeof(int2) * nt) + align256(nt * nt * 256);
}

fa_status fa_prefill_masked(const void* q, const void* k, const void* v, const float* mask, void* out, int B, int T,
                            int Hq, int Hkv, int d, int causal, float scale, float* lse, void* ws, size_t ws_bytes,
                            fa_stream_t stream) {
    set_launch_count(0);
    fa_status st = check_prefill_args(q, k, v, out, B, T, Hq, Hkv, d, scale);
    if (st != FA_OK || B == 0 || T == 0) return st;
    if (!mask) return fa_prefill(q, k, v, out, B, T, Hq, Hkv, d, causal, scale, lse, stream);
    if (!ws || ws_bytes < fa_prefill_masked_workspace_size(T) || (reinterpret_cast<uintptr_t>(ws) & 255))
        return FA_ERR_WORKSPACE;
    if ((st = check_device()) != FA_OK) return st;
    DevCtx ctx;
    if ((st = make_ctx(&ctx)) != FA_OK) return st;
    CUtensorMap tq, tk, tv;
    if ((st = dense_maps(q, k, v, B, T, Hq, Hkv, d, &tq, &tk, &tv)) != FA_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int nt = (T + kTcRows - 1) / kTcRows;
    uint8_t* cls = static_cast<uint8_t*>(ws);
    int32_t* order = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(ws) + align256((size_t)nt * nt));
    int2* range = reinterpret_cast<int2*>(static_cast<uint8_t*>(ws) + align256((size_t)nt * nt) +
                                          align256(sizeof(int32_t) * nt));
    uint8_t* iv = static_cast<uint8_t*>(ws) + align256((size_t)nt * nt) + align256(sizeof(int32_t) * nt) +
                  align256(sizeof(int2) * nt);
    if ((st = launch_mask_classify(mask, T, T, cls, iv, s)) != FA_OK) return st;
    if ((size_t)nt * sizeof(int) > 200 * 1024) return FA_ERR_UNSUPPORTED;
    if (nt * sizeof(int) > 48 * 1024 &&
        (st = raise_dynamic_smem(reinterpret_cast<const void*>(mask_order_kernel), nt * (int)sizeof(int))) != FA_OK)
        return st;
    mask_order_kernel<<<1, 256, nt * sizeof(int), s>>>(cls, nt, nt, causal ? 1 : 0, order, range);
    if (cudaGetLastError() != cudaSuccess) return FA_ERR_CUDA;
    TcParams p = base_params(B, T, Hq, Hkv, causal, scale, out, lse, ctx);
    p.mask = mask;
    p.cls = cls;
    p.iv = iv;
    p.qt_order = order;
    p.qt_range = range;
    p.num_units = dense_units(p);
    const int grid = std::min(p.num_units, sm_count());
    st = launch_tc_d<MODE_MASKED>(d, tq, tk, tv, p, grid, s);
    if (st == FA_OK) set_launch_count(3);
    return st;
}

}  // extern "C"
