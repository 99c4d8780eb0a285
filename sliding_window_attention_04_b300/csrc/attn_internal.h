// Library services shared by the translation units of libswa_attn (not part of the C ABI):
// the lock and device state set up by attn_init, the cached cos/sin tables and the encoding of
// [B, T, H, D] bf16 tensor maps. Implemented in attn_api.cu.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <functional>

namespace swa_host {

struct LibCtx {
  int device;
  int sm_count;
  int* d_err;  // the device error word read by attn_device_status
  PFN_cuTensorMapEncodeTiled_v12000 encode;
};

// Runs f(ctx) with the library lock held and returns its result; ATTN_ERR_NOT_INITIALIZED (without
// calling f) before attn_init or after attn_destroy.
int locked(const std::function<int(const LibCtx&)>& f);

// Inside `locked`: the cached fp32 cos/sin table of (D, base) covering at least T positions, laid out
// [D/4][table_T] of float4 (cos_2m, cos_2m+1, sin_2m, sin_2m+1), and the same entries position-major,
// [table_T][D/4] (`rows`, may be null if not wanted). Returns ATTN_OK or ATTN_ERR_CUDA.
int rope_table_locked(int D, float base, int T, const float4** table, int* table_T, const float4** rows = nullptr);

// The 4-D (d, h, t, b) tensor map of a [B, T, H, D] bf16 tensor whose box is one 128-row tile of one
// head in the tensor core's swizzled layout (64-column boxes for D = 128; rows past T read as zero).
CUresult encode_bf16_tile_map(PFN_cuTensorMapEncodeTiled_v12000 encode, CUtensorMap* map, const void* base, int B,
                              int H, int T, int D);

// Runs f with `dev` as the current device, restoring the caller's device afterwards.
cudaError_t on_device(int dev, const std::function<cudaError_t()>& f);

}  // namespace swa_host
