// Host-side helpers shared by the libfattn translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace fa {

// Device error word of the current device (a file-scope __device__ variable
// in api.cu; its device address is looked up once per device).
unsigned* error_word_ptr(fa_status* st);

// Per-launch device context: error word + current wait bound.
fa_status make_ctx(DevCtx* ctx);

// Number of SMs of the current device (cached per device).
int sm_count();

// Returns FA_OK when the current device is an sm_103 part.
fa_status check_device();

// Raises `kernel`'s dynamic shared-memory limit to at least `bytes` on the
// current device, once per (device, kernel); thread-safe.
fa_status raise_dynamic_smem(const void* kernel, int bytes);

// Records how many kernels the current API call launched (per host thread).
void set_launch_count(int n);

// cuTensorMapEncodeTiled, resolved through the runtime's driver entry point.
fa_status encode_tmap_bf16_4d(CUtensorMap* map, const void* base, const uint64_t dims[4],
                              const uint64_t strides_bytes[3], const uint32_t box[4]);
// 5-D bf16 tensor map, 128-byte swizzle (strides for dims 1..4, in bytes; any order).
fa_status encode_tmap_bf16_5d(CUtensorMap* map, const void* base, const uint64_t dims[5], const uint64_t strides_bytes[4],
                              const uint32_t box[5]);
// The same for any element type and swizzle mode.
fa_status encode_tmap_4d(CUtensorMap* map, const void* base, const uint64_t dims[4], const uint64_t strides_bytes[3],
                         const uint32_t box[4], CUtensorMapDataType dtype, CUtensorMapSwizzle swizzle);

// Prefill of query rows [q0, q0 + Tq) of every sequence against keys [0, Tk)
// (defined in attn_tc.cu; used by the host-buffer pipeline).
fa_status launch_prefill_rows(const void* q, const void* k, const void* v, void* out, int B, int T, int Hq, int Hkv,
                              int d, int causal, float scale, int q0, int Tq, int Tk, cudaStream_t s);

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool aligned32(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 31u) == 0; }

inline fa_status cuda_status(cudaError_t e) { return e == cudaSuccess ? FA_OK : FA_ERR_CUDA; }

}  // namespace fa
