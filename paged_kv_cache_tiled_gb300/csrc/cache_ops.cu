// Memory-bound helper kernels of libfattn:
//   * fused KV-cache append ("Fast Attention Kernels and Operator Fusion",
//     section "Operator Fusion", fusion list: updating the KV cache while
//     transforming key and value tensors), and its variant that also applies
//     rotary position embeddings to queries and keys (same list);
//   * fp32 -> bf16 staging cast;
//   * block-table gather test hook ("Paged Attention Kernels": translate each
//     logical position through the block table);
//   * additive-mask tile classifier used by the masked prefill
//     ("FlashAttention-Style Kernels", attention equation with additive M).
// All of them move data with 16-byte vector accesses and are sized by
// grid-stride loops over a multiple of the SM count.
#include "host_common.cuh"

namespace fa {

constexpr int kBlock = 16;  // tokens per cache block

// ------------------------------------------------------------ append ------
// One thread moves one 16-byte chunk (8 bf16) of one (token, head) row of K
// and the same chunk of V.  Input rows are contiguous [N, Hkv, d]; the cache
// row of (slot, head) starts at ((slot/16 * Hkv + head) * 16 + slot%16) * d.
template <bool kF32>
__global__ void __launch_bounds__(256) cache_append_kernel(const void* __restrict__ k, const void* __restrict__ v,
                                                           uint16_t* __restrict__ kc, uint16_t* __restrict__ vc,
                                                           const int32_t* __restrict__ slots, int N, int Hkv,
                                                           int d, int num_blocks, DevCtx ctx) {
    const int cpr = d >> 3;  // chunks per row
    const long total = (long)N * Hkv * cpr;
    for (long idx = (long)blockIdx.x * blockDim.x + threadIdx.x; idx < total; idx += (long)gridDim.x * blockDim.x) {
        const int c = (int)(idx % cpr);
        const long row = idx / cpr;  // token * Hkv + head
        const int h = (int)(row % Hkv);
        const long tok = row / Hkv;
        const int slot = __ldg(slots + tok);
        if (slot < 0) continue;
        if (slot >= num_blocks * kBlock) {
            raise_error(ctx, ERR_BOUNDS_BIT);
            continue;
        }
        const long dst = (((long)(slot / kBlock) * Hkv + h) * kBlock + (slot % kBlock)) * d + c * 8;
        uint4 kv4, vv4;
        if constexpr (kF32) {
            const float4* ks = reinterpret_cast<const float4*>(static_cast<const float*>(k) + row * d + c * 8);
            const float4* vs = reinterpret_cast<const float4*>(static_cast<const float*>(v) + row * d + c * 8);
            float4 a = __ldg(ks), b = __ldg(ks + 1), e = __ldg(vs), f = __ldg(vs + 1);
            kv4 = make_uint4(pack_bf16x2(a.x, a.y), pack_bf16x2(a.z, a.w), pack_bf16x2(b.x, b.y),
                             pack_bf16x2(b.z, b.w));
            vv4 = make_uint4(pack_bf16x2(e.x, e.y), pack_bf16x2(e.z, e.w), pack_bf16x2(f.x, f.y),
                             pack_bf16x2(f.z, f.w));
        } else {
            kv4 = __ldg(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(k) + row * d + c * 8));
            vv4 = __ldg(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(v) + row * d + c * 8));
        }
        *reinterpret_cast<uint4*>(kc + dst) = kv4;
        *reinterpret_cast<uint4*>(vc + dst) = vv4;
    }
}

// ------------------------------------------------------ rotary append ----
// Rotate-half rotary embedding: channel j pairs with j + d/2 and turns by the
// angle whose cosine / sine sit at columns j / d/2 + j of row `pos` of the
// caller's fp32 table:  y_j = x_j c - x_{j+d/2} s,  y_{j+d/2} = x_{j+d/2} c + x_j s
// (fp32, rounded once to bf16).  One thread handles 8 channel pairs of one
// row: the 16-byte chunk at channel 8c and its partner chunk at d/2 + 8c.
// Rows of a token: its Hq query rows (rotated into q_out), then its Hkv key
// rows (rotated into the cache slot); the thread of a key chunk pair also
// copies the same two chunks of the value row.
template <bool kF32>
__device__ __forceinline__ void load8(const void* base, long off, float (&x)[8]) {
    if constexpr (kF32) {
        const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(base) + off);
        const float4 a = __ldg(p), b = __ldg(p + 1);
        x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w; x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
    } else {
        const uint4 u = __ldg(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(base) + off));
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            x[2 * i] = __uint_as_float(w[i] << 16);
            x[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
        }
    }
}
__device__ __forceinline__ uint4 pack8(const float (&y)[8]) {
    return make_uint4(pack_bf16x2(y[0], y[1]), pack_bf16x2(y[2], y[3]), pack_bf16x2(y[4], y[5]),
                      pack_bf16x2(y[6], y[7]));
}

template <bool kF32>
__global__ void __launch_bounds__(256) rope_append_kernel(const void* __restrict__ q, const void* __restrict__ k,
                                                          const void* __restrict__ v,
                                                          const int32_t* __restrict__ positions,
                                                          const float* __restrict__ cos_sin, int max_pos,
                                                          uint16_t* __restrict__ q_out, uint16_t* __restrict__ kc,
                                                          uint16_t* __restrict__ vc,
                                                          const int32_t* __restrict__ slots, int N, int Hq, int Hkv,
                                                          int d, int num_blocks, DevCtx ctx) {
    const int half = d >> 1, cph = half >> 3;  // chunk pairs per row
    const int rpt = Hq + Hkv;                   // rotated rows per token
    const long total = (long)N * rpt * cph;
    for (long idx = (long)blockIdx.x * blockDim.x + threadIdx.x; idx < total; idx += (long)gridDim.x * blockDim.x) {
        const int c = (int)(idx % cph);
        const long row = idx / cph;
        const long tok = row / rpt;
        const int r = (int)(row % rpt);
        const int pos = __ldg(positions + tok);
        if (pos < 0 || pos >= max_pos) {
            raise_error(ctx, ERR_BOUNDS_BIT);
            continue;
        }
        const bool is_q = r < Hq;
        const int h = is_q ? r : r - Hq;
        long dst = 0;
        if (!is_q) {
            const int slot = __ldg(slots + tok);
            if (slot < 0) continue;
            if (slot >= num_blocks * kBlock) {
                raise_error(ctx, ERR_BOUNDS_BIT);
                continue;
            }
            dst = (((long)(slot / kBlock) * Hkv + h) * kBlock + (slot % kBlock)) * d;
        }
        const long src = is_q ? (tok * Hq + h) * d : (tok * Hkv + h) * d;
        float x1[8], x2[8], co[8], si[8], y1[8], y2[8];
        load8<kF32>(is_q ? q : k, src + c * 8, x1);
        load8<kF32>(is_q ? q : k, src + half + c * 8, x2);
        const float4* cs = reinterpret_cast<const float4*>(cos_sin + (long)pos * d + c * 8);
        const float4* sn = reinterpret_cast<const float4*>(cos_sin + (long)pos * d + half + c * 8);
        const float4 c0 = __ldg(cs), c1 = __ldg(cs + 1), s0 = __ldg(sn), s1 = __ldg(sn + 1);
        co[0] = c0.x; co[1] = c0.y; co[2] = c0.z; co[3] = c0.w; co[4] = c1.x; co[5] = c1.y; co[6] = c1.z; co[7] = c1.w;
        si[0] = s0.x; si[1] = s0.y; si[2] = s0.z; si[3] = s0.w; si[4] = s1.x; si[5] = s1.y; si[6] = s1.z; si[7] = s1.w;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            y1[i] = fmaf(x1[i], co[i], -(x2[i] * si[i]));
            y2[i] = fmaf(x2[i], co[i], x1[i] * si[i]);
        }
        if (is_q) {
            *reinterpret_cast<uint4*>(q_out + src + c * 8) = pack8(y1);
            *reinterpret_cast<uint4*>(q_out + src + half + c * 8) = pack8(y2);
        } else {
            *reinterpret_cast<uint4*>(kc + dst + c * 8) = pack8(y1);
            *reinterpret_cast<uint4*>(kc + dst + half + c * 8) = pack8(y2);
            float v1[8], v2[8];
            load8<kF32>(v, src + c * 8, v1);
            load8<kF32>(v, src + half + c * 8, v2);
            *reinterpret_cast<uint4*>(vc + dst + c * 8) = pack8(v1);
            *reinterpret_cast<uint4*>(vc + dst + half + c * 8) = pack8(v2);
        }
    }
}

// ------------------------------------------------------- 8-bit append -----
// One thread quantises 16 channels of one (token, head) row of K and of V:
// code = E4M3(x / scale) (binary32 division, round to nearest even,
// saturating).  K codes are one 16-byte store into the row [blk][h][off];
// V codes go to the channel-major block [blk][h][c][off], one byte per channel.
template <bool kF32>
__global__ void __launch_bounds__(256) cache_append_fp8_kernel(const void* __restrict__ k, const void* __restrict__ v,
                                                               uint8_t* __restrict__ kc, uint8_t* __restrict__ vc,
                                                               const int32_t* __restrict__ slots, int N, int Hkv, int d,
                                                               int num_blocks, float k_scale, float v_scale,
                                                               DevCtx ctx) {
    const int cpr = d >> 4;  // 16-channel chunks per row
    const long total = (long)N * Hkv * cpr;
    for (long idx = (long)blockIdx.x * blockDim.x + threadIdx.x; idx < total; idx += (long)gridDim.x * blockDim.x) {
        const int c = (int)(idx % cpr);
        const long row = idx / cpr;
        const int h = (int)(row % Hkv);
        const long tok = row / Hkv;
        const int slot = __ldg(slots + tok);
        if (slot < 0) continue;
        if (slot >= num_blocks * kBlock) {
            raise_error(ctx, ERR_BOUNDS_BIT);
            continue;
        }
        const long blk = slot / kBlock, off = slot % kBlock;
        float x[16], y[16];
        load8<kF32>(k, row * d + c * 16, *reinterpret_cast<float(*)[8]>(x));
        load8<kF32>(k, row * d + c * 16 + 8, *reinterpret_cast<float(*)[8]>(x + 8));
        load8<kF32>(v, row * d + c * 16, *reinterpret_cast<float(*)[8]>(y));
        load8<kF32>(v, row * d + c * 16 + 8, *reinterpret_cast<float(*)[8]>(y + 8));
        uint32_t kw[4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
            kw[i] = f32x2_to_e4m3x2(__fdiv_rn(x[4 * i], k_scale), __fdiv_rn(x[4 * i + 1], k_scale)) |
                    (f32x2_to_e4m3x2(__fdiv_rn(x[4 * i + 2], k_scale), __fdiv_rn(x[4 * i + 3], k_scale)) << 16);
        *reinterpret_cast<uint4*>(kc + ((blk * Hkv + h) * kBlock + off) * d + c * 16) =
            make_uint4(kw[0], kw[1], kw[2], kw[3]);
        uint8_t* vrow = vc + ((blk * Hkv + h) * d + c * 16) * kBlock + off;
#pragma unroll
        for (int i = 0; i < 16; i += 2) {
            const uint32_t b = f32x2_to_e4m3x2(__fdiv_rn(y[i], v_scale), __fdiv_rn(y[i + 1], v_scale));
            vrow[i * kBlock] = (uint8_t)(b & 0xFF);
            vrow[(i + 1) * kBlock] = (uint8_t)(b >> 8);
        }
    }
}

// -------------------------------------------------------- block copy ------
// Copy-on-write for the block pool: pair i copies physical block
// pairs[2i] onto pairs[2i+1] in both caches (Hkv * 16 * d bf16 each),
// 16 bytes per thread.
__global__ void __launch_bounds__(256) copy_blocks_kernel(uint16_t* __restrict__ kc, uint16_t* __restrict__ vc,
                                                          const int32_t* __restrict__ pairs, int n, int Hkv, int d,
                                                          int num_blocks, DevCtx ctx) {
    const long per = (long)Hkv * kBlock * d / 8;  // 16-byte chunks per block
    const long total = (long)n * per;
    for (long idx = (long)blockIdx.x * blockDim.x + threadIdx.x; idx < total; idx += (long)gridDim.x * blockDim.x) {
        const long i = idx / per, c = idx % per;
        const int src = __ldg(pairs + 2 * i), dst = __ldg(pairs + 2 * i + 1);
        if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
            raise_error(ctx, ERR_BOUNDS_BIT);
            continue;
        }
        const long so = (long)src * per + c, dof = (long)dst * per + c;
        reinterpret_cast<uint4*>(kc)[dof] = reinterpret_cast<const uint4*>(kc)[so];
        reinterpret_cast<uint4*>(vc)[dof] = reinterpret_cast<const uint4*>(vc)[so];
    }
}

// ------------------------------------------------------------- stage ------
__global__ void __launch_bounds__(256) stage_bf16_kernel(const float* __restrict__ src, uint16_t* __restrict__ dst,
                                                         size_t n) {
    const size_t n8 = n / 8;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n8; i += (size_t)gridDim.x * blockDim.x) {
        const float4* s = reinterpret_cast<const float4*>(src) + 2 * i;
        float4 a = __ldg(s), b = __ldg(s + 1);
        *reinterpret_cast<uint4*>(dst + 8 * i) =
            make_uint4(pack_bf16x2(a.x, a.y), pack_bf16x2(a.z, a.w), pack_bf16x2(b.x, b.y), pack_bf16x2(b.z, b.w));
    }
    if (blockIdx.x == 0)
        for (size_t i = n8 * 8 + threadIdx.x; i < n; i += blockDim.x) {
            __nv_bfloat16 b = __float2bfloat16_rn(src[i]);
            dst[i] = *reinterpret_cast<uint16_t*>(&b);
        }
}

// ------------------------------------------------------------ gather ------
__global__ void __launch_bounds__(256) gather_kv_kernel(const uint16_t* __restrict__ cache,
                                                        const int32_t* __restrict__ bt,
                                                        const int32_t* __restrict__ ctx_lens,
                                                        uint16_t* __restrict__ out, int num_seqs, int mbps,
                                                        int num_blocks, int Hkv, int d, int max_ctx, DevCtx ctx) {
    const int cpr = d >> 3;
    const long per_seq = (long)max_ctx * Hkv * cpr;
    const long total = per_seq * num_seqs;
    for (long idx = (long)blockIdx.x * blockDim.x + threadIdx.x; idx < total; idx += (long)gridDim.x * blockDim.x) {
        const int s = (int)(idx / per_seq);
        const long r = idx % per_seq;
        const int c = (int)(r % cpr);
        const int h = (int)((r / cpr) % Hkv);
        const int t = (int)(r / ((long)cpr * Hkv));
        const int L = __ldg(ctx_lens + s);
        if (t >= L) continue;
        if (L > mbps * kBlock) {
            raise_error(ctx, ERR_BOUNDS_BIT);
            continue;
        }
        const int phys = __ldg(bt + (long)s * mbps + t / kBlock);
        if (phys < 0 || phys >= num_blocks) {
            raise_error(ctx, ERR_BOUNDS_BIT);
            continue;
        }
        const long src = (((long)phys * Hkv + h) * kBlock + t % kBlock) * d + c * 8;
        const long dst = (((long)s * max_ctx + t) * Hkv + h) * d + c * 8;
        *reinterpret_cast<uint4*>(out + dst) = __ldg(reinterpret_cast<const uint4*>(cache + src));
    }
}

// ------------------------------------------------------- mask classes -----
// One CTA per 128x128 tile of the mask (edge tiles: their in-range elements):
// class 0 when every element is -inf, 1 when every element is exactly 0, 3
// when every element is 0 or -inf and the zeros of each row are one
// contiguous run (possibly empty) -- the tile only restricts each query row to
// an interval of keys -- and 2 otherwise.  For a class-3 tile, iv (when not
// null) gets each of the 128 rows' run [lo, hi) as two bytes, at
// iv[((ti * ntj + tj) * 128 + r) * 2] (rows past Tq, and rows without a zero,
// get 0, 0).  Every tile is read once with coalesced 16-byte loads when the
// row length allows; only the tiles of 0 and -inf that are neither all 0 nor
// all -inf are read a second time, row by row, for the runs.
__global__ void __launch_bounds__(256) mask_classify_kernel(const float* __restrict__ M, int Tq, int Tk,
                                                            uint8_t* __restrict__ cls, uint8_t* __restrict__ iv) {
    __shared__ uint8_t run[128][2];
    const int tj = blockIdx.x, ti = blockIdx.y;
    const int i0 = ti * 128, j0 = tj * 128;
    const int rows = min(128, Tq - i0), cols = min(128, Tk - j0);
    const int lane = threadIdx.x & 31, rgrp = threadIdx.x >> 5;
    const bool vec = (Tk % 4 == 0) && (cols == 128);
    // pass 1: is every element -inf, is every element 0, is any element
    // neither (one read of the tile)
    bool all_ninf = true, all_zero = true, only_0_inf = true;
    auto take = [&](float x) {
        all_ninf &= (x == -INFINITY);
        all_zero &= (x == 0.f);
        only_0_inf &= (x == 0.f) | (x == -INFINITY);
    };
    if (vec) {
        // 32 threads cover one 512-byte row; 8 rows per pass
        for (int r = rgrp; r < rows; r += 8) {
            const float4 x = __ldg(reinterpret_cast<const float4*>(M + (long)(i0 + r) * Tk + j0) + lane);
            take(x.x);
            take(x.y);
            take(x.z);
            take(x.w);
        }
    } else {
        for (int e = threadIdx.x; e < rows * cols; e += blockDim.x) take(__ldg(M + (long)(i0 + e / cols) * Tk + j0 + e % cols));
    }
    const int n_inf = __syncthreads_and(all_ninf);
    const int n_zero = __syncthreads_and(all_zero);
    const int n_01 = __syncthreads_and(only_0_inf);
    uint8_t c = (uint8_t)(n_inf ? 0 : (n_zero ? 1 : 2));
    if (c == 2 && n_01) {
        // pass 2 (tiles of 0 and -inf only, both present): one warp per row
        // re-reads the row (from L2) and finds its first and last zero and the
        // number of zeros; the row keeps one run of keys when they agree
        bool runs = true;
        for (int r = rgrp; r < 128; r += 8) {
            int lo = 0, hi = 0;
            if (r < rows) {
                int zeros = 0, first = 128, last = -1;
                for (int j = lane; j < cols; j += 32)
                    if (__ldg(M + (long)(i0 + r) * Tk + j0 + j) == 0.f) {
                        first = min(first, j);
                        last = j;
                        ++zeros;
                    }
                zeros = __reduce_add_sync(0xffffffffu, zeros);
                if (zeros > 0) {
                    lo = __reduce_min_sync(0xffffffffu, first);
                    hi = __reduce_max_sync(0xffffffffu, last) + 1;
                    runs &= zeros == hi - lo;
                }
            }
            if (lane == 0) {
                run[r][0] = (uint8_t)lo;
                run[r][1] = (uint8_t)hi;
            }
        }
        if (__syncthreads_and(runs)) c = 3;
    }
    const long tile = (long)ti * gridDim.x + tj;
    if (threadIdx.x == 0) cls[tile] = c;
    if (c == 3 && iv)
        for (int e = threadIdx.x; e < 256; e += blockDim.x) iv[tile * 256 + e] = run[e >> 1][e & 1];
}

// Launched from the masked prefill entry point.
fa_status launch_mask_classify(const float* M, int Tq, int Tk, uint8_t* cls, uint8_t* iv, cudaStream_t s) {
    dim3 grid((Tk + 127) / 128, (Tq + 127) / 128);
    mask_classify_kernel<<<grid, 256, 0, s>>>(M, Tq, Tk, cls, iv);
    return cuda_status(cudaGetLastError());
}

static int grid_for(long work, int per_cta) {
    long g = (work + per_cta - 1) / per_cta;
    long cap = (long)sm_count() * 8;
    if (g > cap) g = cap;
    return (int)(g < 1 ? 1 : g);
}

}  // namespace fa

using namespace fa;

extern "C" {

fa_status fa_cache_append(const void* k, const void* v, void* k_cache, void* v_cache, const int32_t* slot_mapping,
                          int N, int Hkv, int d, int num_blocks, fa_dtype in_dtype, fa_stream_t stream) {
    set_launch_count(0);
    if (N < 0 || Hkv <= 0 || num_blocks < 0) return FA_ERR_INVALID_ARG;
    if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
    if (in_dtype != FA_BF16 && in_dtype != FA_F32) return FA_ERR_INVALID_ARG;
    if (N == 0) return FA_OK;
    if (!k || !v || !k_cache || !v_cache || !slot_mapping) return FA_ERR_INVALID_ARG;
    if (!aligned16(k) || !aligned16(v) || !aligned16(k_cache) || !aligned16(v_cache)) return FA_ERR_INVALID_ARG;
    fa_status st = check_device();
    if (st != FA_OK) return st;
    DevCtx ctx;
    if ((st = make_ctx(&ctx)) != FA_OK) return st;
    const long work = (long)N * Hkv * (d / 8);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (in_dtype == FA_F32)
        cache_append_kernel<true><<<grid_for(work, 256), 256, 0, s>>>(k, v, static_cast<uint16_t*>(k_cache),
                                                                      static_cast<uint16_t*>(v_cache), slot_mapping,
                                                                      N, Hkv, d, num_blocks, ctx);
    else
        cache_append_kernel<false><<<grid_for(work, 256), 256, 0, s>>>(k, v, static_cast<uint16_t*>(k_cache),
                                                                       static_cast<uint16_t*>(v_cache),
                                                                       slot_mapping, N, Hkv, d, num_blocks, ctx);
    st = cuda_status(cudaGetLastError());
    if (st == FA_OK) set_launch_count(1);
    return st;
}

fa_status fa_mask_tile_classes(const float* mask, int Tq, int Tk, uint8_t* cls, uint8_t* intervals,
                               fa_stream_t stream) {
    set_launch_count(0);
    if (Tq < 0 || Tk < 0) return FA_ERR_INVALID_ARG;
    if (Tq == 0 || Tk == 0) return FA_OK;
    if (!mask || !cls || !aligned16(mask)) return FA_ERR_INVALID_ARG;
    if ((Tq + 127) / 128 > 65535) return FA_ERR_UNSUPPORTED;  // grid y limit
    fa_status st = check_device();
    if (st != FA_OK) return st;
    st = launch_mask_classify(mask, Tq, Tk, cls, intervals, reinterpret_cast<cudaStream_t>(stream));
    if (st == FA_OK) set_launch_count(1);
    return st;
}

fa_status fa_stage_bf16(const float* src, void* dst, size_t n, fa_stream_t stream) {
    set_launch_count(0);
    if (n == 0) return FA_OK;
    if (!src || !dst || !aligned16(src) || !aligned16(dst)) return FA_ERR_INVALID_ARG;
    fa_status st = check_device();
    if (st != FA_OK) return st;
    stage_bf16_kernel<<<grid_for((long)(n / 8 + 1), 256), 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        src, static_cast<uint16_t*>(dst), n);
    st = cuda_status(cudaGetLastError());
    if (st == FA_OK) set_launch_count(1);
    return st;
}

fa_status fa_debug_gather_kv(const void* cache, const int32_t* block_table, const int32_t* ctx_lens, void* out,
                             int num_seqs, int max_blocks_per_seq, int num_blocks, int Hkv, int d, int max_ctx,
                             fa_stream_t stream) {
    set_launch_count(0);
    if (num_seqs < 0 || max_blocks_per_seq < 0 || num_blocks < 0 || Hkv <= 0 || max_ctx < 0)
        return FA_ERR_INVALID_ARG;
    if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
    if (num_seqs == 0 || max_ctx == 0) return FA_OK;
    if (!cache || !block_table || !ctx_lens || !out || !aligned16(cache) || !aligned16(out))
        return FA_ERR_INVALID_ARG;
    fa_status st = check_device();
    if (st != FA_OK) return st;
    DevCtx ctx;
    if ((st = make_ctx(&ctx)) != FA_OK) return st;
    const long work = (long)num_seqs * max_ctx * Hkv * (d / 8);
    gather_kv_kernel<<<grid_for(work, 256), 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint16_t*>(cache), block_table, ctx_lens, static_cast<uint16_t*>(out), num_seqs,
        max_blocks_per_seq, num_blocks, Hkv, d, max_ctx, ctx);
    st = cuda_status(cudaGetLastError());
    if (st == FA_OK) set_launch_count(1);
    return st;
}

fa_status fa_cache_append_rope(const void* q, const void* k, const void* v, const int32_t* positions,
                               const float* cos_sin, int max_pos, void* q_out, void* k_cache, void* v_cache,
                               const int32_t* slot_mapping, int N, int Hq, int Hkv, int d, int num_blocks,
                               fa_dtype in_dtype, fa_stream_t stream) {
    set_launch_count(0);
    if (N < 0 || Hq <= 0 || Hkv <= 0 || num_blocks < 0 || max_pos <= 0) return FA_ERR_INVALID_ARG;
    if (in_dtype != FA_BF16 && in_dtype != FA_F32) return FA_ERR_INVALID_ARG;
    if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
    if (N == 0) return FA_OK;
    if (!q || !k || !v || !positions || !cos_sin || !q_out || !k_cache || !v_cache || !slot_mapping)
        return FA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(cos_sin) || !aligned16(q_out) ||
        !aligned16(k_cache) || !aligned16(v_cache))
        return FA_ERR_INVALID_ARG;
    fa_status st = check_device();
    if (st != FA_OK) return st;
    DevCtx ctx;
    if ((st = make_ctx(&ctx)) != FA_OK) return st;
    const long work = (long)N * (Hq + Hkv) * (d / 16);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (in_dtype == FA_F32)
        rope_append_kernel<true><<<grid_for(work, 256), 256, 0, s>>>(
            q, k, v, positions, cos_sin, max_pos, static_cast<uint16_t*>(q_out), static_cast<uint16_t*>(k_cache),
            static_cast<uint16_t*>(v_cache), slot_mapping, N, Hq, Hkv, d, num_blocks, ctx);
    else
        rope_append_kernel<false><<<grid_for(work, 256), 256, 0, s>>>(
            q, k, v, positions, cos_sin, max_pos, static_cast<uint16_t*>(q_out), static_cast<uint16_t*>(k_cache),
            static_cast<uint16_t*>(v_cache), slot_mapping, N, Hq, Hkv, d, num_blocks, ctx);
    st = cuda_status(cudaGetLastError());
    if (st == FA_OK) set_launch_count(1);
    return st;
}

fa_status fa_cache_append_fp8(const void* k, const void* v, void* k_cache, void* v_cache, const int32_t* slot_mapping,
                              int N, int Hkv, int d, int num_blocks, float k_scale, float v_scale, fa_dtype in_dtype,
                              fa_stream_t stream) {
    set_launch_count(0);
    if (N < 0 || Hkv <= 0 || num_blocks < 0 || !(k_scale > 0.f) || !(k_scale < INFINITY) || !(v_scale > 0.f) ||
        !(v_scale < INFINITY))
        return FA_ERR_INVALID_ARG;
    if (in_dtype != FA_BF16 && in_dtype != FA_F32) return FA_ERR_INVALID_ARG;
    if (d != 128) return FA_ERR_UNSUPPORTED;
    if (N == 0) return FA_OK;
    if (!k || !v || !k_cache || !v_cache || !slot_mapping || !aligned16(k) || !aligned16(v) || !aligned16(k_cache) ||
        !aligned16(v_cache))
        return FA_ERR_INVALID_ARG;
    fa_status st = check_device();
    if (st != FA_OK) return st;
    DevCtx ctx;
    if ((st = make_ctx(&ctx)) != FA_OK) return st;
    const long work = (long)N * Hkv * (d / 16);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (in_dtype == FA_F32)
        cache_append_fp8_kernel<true><<<grid_for(work, 256), 256, 0, s>>>(
            k, v, static_cast<uint8_t*>(k_cache), static_cast<uint8_t*>(v_cache), slot_mapping, N, Hkv, d,
            num_blocks, k_scale, v_scale, ctx);
    else
        cache_append_fp8_kernel<false><<<grid_for(work, 256), 256, 0, s>>>(
            k, v, static_cast<uint8_t*>(k_cache), static_cast<uint8_t*>(v_cache), slot_mapping, N, Hkv, d,
            num_blocks, k_scale, v_scale, ctx);
    st = cuda_status(cudaGetLastError());
    if (st == FA_OK) set_launch_count(1);
    return st;
}

fa_status fa_copy_blocks(void* k_cache, void* v_cache, const int32_t* pairs, int n, int Hkv, int d, int num_blocks,
                         fa_stream_t stream) {
    set_launch_count(0);
    if (n < 0 || Hkv <= 0 || num_blocks < 0) return FA_ERR_INVALID_ARG;
    if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
    if (n == 0) return FA_OK;
    if (!k_cache || !v_cache || !pairs || !aligned16(k_cache) || !aligned16(v_cache)) return FA_ERR_INVALID_ARG;
    fa_status st = check_device();
    if (st != FA_OK) return st;
    DevCtx ctx;
    if ((st = make_ctx(&ctx)) != FA_OK) return st;
    const long work = (long)n * Hkv * kBlock * d / 8;
    copy_blocks_kernel<<<grid_for(work, 256), 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        static_cast<uint16_t*>(k_cache), static_cast<uint16_t*>(v_cache), pairs, n, Hkv, d, num_blocks, ctx);
    st = cuda_status(cudaGetLastError());
    if (st == FA_OK) set_launch_count(1);
    return st;
}

}  // extern "C"
