// Shared definitions of the attention forward kernels: launch parameters, the operand tile
// layout in shared memory, the QK-norm + RoPE row transform and the mask predicate.
#pragma once
#include <cstdint>
#include <cuda_bf16.h>

#include "ptx.cuh"

namespace swa {

constexpr int kTile = 128;  // rows of a Q tile and keys of a K/V tile

// Device-side error codes written to the error word (host maps them to ATTN_ERR_*).
constexpr int kDevErrTimeout = 1;

struct AttnParams {
  const __nv_bfloat16* q;  // [B, T, H, D]
  const __nv_bfloat16* k;  // [B, T, H, D]
  const __nv_bfloat16* v;  // [B, T, H, D]
  __nv_bfloat16* out;      // [B, T, H, D]
  float* lse;              // [B, H, T] or nullptr
  const float2* rope;      // [T_table, D/2] (cos, sin) or nullptr (RoPE off)
  int* err;                // device error word
  int B, H, T;
  int window;              // < 0: no window
  int causal;
  int use_norm;
  float eps;
  float scale_log2;        // log2(e) / sqrt(D)
  int n_qtiles;            // ceil(T / 128)
};

// Byte offset of 16-byte chunk `chunk` (8 bf16 along D) of row `row` inside a 128-row operand
// tile stored the way the tensor core reads a K-major (row = M or N index, D contiguous) bf16
// tile with the 128-byte swizzle (D >= 64: sub-tiles of 64 columns, 16 KB apart) or the 64-byte
// swizzle (D = 32). The same physical layout serves V as an MN-major B operand (row = key).
template <int D>
__device__ __forceinline__ uint32_t tile_off(int row, int chunk) {
  if constexpr (D >= 64) {
    const int sub = chunk >> 3, c = chunk & 7;
    return static_cast<uint32_t>(sub * (kTile * 128) + row * 128 + ((c ^ (row & 7)) << 4));
  } else {
    return static_cast<uint32_t>(row * 64 + ((chunk ^ ((row >> 1) & 3)) << 4));
  }
}

template <int D>
struct TileGeom {
  static constexpr int kBytes = kTile * D * 2;             // one 128 x D bf16 tile
  static constexpr int kRowBytes = D >= 64 ? 128 : 64;     // bytes of a row inside a sub-tile
  static constexpr uint32_t kSwizzle = D >= 64 ? 2u : 4u;  // descriptor swizzle mode
  static constexpr uint32_t kSBO = 8 * kRowBytes;          // stride between 8-row groups
  static constexpr int kKSteps = D / 16;                   // UMMA K steps over D
  // start byte offset of UMMA K step `ks` (16 elements along D) within a K-major tile
  static __device__ __forceinline__ uint32_t kstep_off(int ks) {
    if constexpr (D >= 64) return static_cast<uint32_t>((ks >> 2) * (kTile * 128) + (ks & 3) * 32);
    else return static_cast<uint32_t>(ks * 32);
  }
};

// Is key j visible to query i?  FlashAttention window convention: window_size = (W, 0) for
// causal, (W, W) otherwise; W < 0 means unbounded.
__device__ __forceinline__ bool key_visible(int i, int j, int T, int window, int causal) {
  if (j >= T) return false;
  if (causal && j > i) return false;
  if (window >= 0) {
    if (j < i - window) return false;
    if (!causal && j > i + window) return false;
  }
  return true;
}

// QK-norm + RoPE for one row held in registers as fp32 x[0..D):
//   r = 1 / sqrt(mean(x^2) + eps)   (parameter-free RMSNorm; r = 1 when !use_norm)
//   pair i = (x[i], x[i + D/2]) at position pos, angle pos * base^(-2i/D) from the table:
//   y[i] = x1 (c r) + x2 (s r),  y[i + D/2] = x2 (c r) - x1 (s r)
// The result is rounded to bf16 (a quantisation), so the fp32 evaluation is pinned to one fixed
// sequence of correctly rounded operations: the sum of squares accumulates d = 0..D-1 with
// fused multiply-adds, r is a rounded square root followed by a rounded division, and every
// product / fused multiply-add is spelled out with the _rn intrinsics so the compiler cannot
// re-associate or contract them.
// The bf16 result is written as D/8 16-byte chunks through `store(chunk, uint4)`.
template <int D, typename Store>
__device__ __forceinline__ void qk_row_transform(float (&x)[D], int pos, const float2* rope, int use_norm,
                                                 float eps, Store store) {
  float r = 1.0f;
  if (use_norm) {
    float ss = 0.f;
#pragma unroll
    for (int d = 0; d < D; ++d) ss = __fmaf_rn(x[d], x[d], ss);
    const float ms = __fmul_rn(ss, 1.0f / D);
    r = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(ms, eps)));
  }
  constexpr int H2 = D / 2;
  if (rope != nullptr) {
    const float2* cs = rope + static_cast<size_t>(pos) * H2;
#pragma unroll
    for (int i = 0; i < H2; ++i) {
      const float2 t = __ldg(cs + i);
      const float c = __fmul_rn(t.x, r), s = __fmul_rn(t.y, r);
      const float x1 = x[i], x2 = x[i + H2];
      x[i] = __fmaf_rn(x1, c, __fmul_rn(x2, s));
      x[i + H2] = __fmaf_rn(x2, c, -__fmul_rn(x1, s));
    }
  } else {
#pragma unroll
    for (int d = 0; d < D; ++d) x[d] = __fmul_rn(x[d], r);
  }
#pragma unroll
  for (int ch = 0; ch < D / 8; ++ch) {
    uint4 u;
    u.x = pack_bf16x2(x[ch * 8 + 0], x[ch * 8 + 1]);
    u.y = pack_bf16x2(x[ch * 8 + 2], x[ch * 8 + 3]);
    u.z = pack_bf16x2(x[ch * 8 + 4], x[ch * 8 + 5]);
    u.w = pack_bf16x2(x[ch * 8 + 6], x[ch * 8 + 7]);
    store(ch, u);
  }
}

__device__ __forceinline__ void bf16x8_to_f32(const uint4 u, float* f) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

__device__ __forceinline__ void report_error(int* err, int code) {
  if (err != nullptr) atomicCAS(err, 0, code);
}

}  // namespace swa
