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
  const __nv_bfloat16* k;  // [B, T, Hkv, D]
  const __nv_bfloat16* v;  // [B, T, Hkv, D]
  __nv_bfloat16* out;      // [B, T, H, D]
  float* lse;              // [B, H, T] or nullptr
  const float4* rope;      // [D/4][rope_T] (cos_2i, cos_2i+1, sin_2i, sin_2i+1), or nullptr (RoPE off)
  int rope_T;              // positions the table covers (its row stride), >= T
  int* err;                // device error word
  int B, H, T;
  int Hkv;                 // K/V heads; query head h uses K/V head h / kv_group
  int kv_group;            // H / Hkv (1: multi-head attention)
  int window;              // < 0: no window
  int causal;
  int use_norm;
  float eps;
  float scale_log2;        // log2(e) / sqrt(D)
  float ref_log2;          // > 0: a bound on every scaled score (log2 units), used as a fixed softmax
                           // reference; 0: no bound known (QK-norm off), running maximum instead
  int n_qtiles;            // ceil(T / 128)
  int head_group;          // persistent kernel: heads per ticket group (their K/V fit in L2 together)
  int n_long;              // persistent kernel: heads 0 .. n_long - 1 run as one ticket each (all their
                           // query blocks); the others as tickets of two query blocks
  // value-embedding gate (nullptr ve: none): v <- v + gate[b, t, hk] ve, where the gate factor
  // 2 sigmoid(xg[b, t, 0:32] . wg[hk, 0:32]) is computed once per (b, t, hk) by ve_gate_kernel
  const __nv_bfloat16* ve;  // [B, T, Hkv, D]
  const __nv_bfloat16* xg;  // rows of xg_stride elements, [B, T, xg_stride]; the first 32 are used
  const __nv_bfloat16* wg;  // [Hkv, 32]
  int xg_stride;
  float* gate;              // [B, T, Hkv] gate factors (caller's workspace)
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

// QK-norm + RoPE for one row of D bf16 values held as D/2 packed words w (element 2k in the
// low half of w[k]), transformed in place:
//   r = 1 / sqrt(mean(x^2) + eps)   (parameter-free RMSNorm; r = 1 when !use_norm)
//   pair i = (x[i], x[i + D/2]) at position pos, angle pos * base^(-2i/D) from the table:
//   y[i] = x1 (c r) + x2 (s r),  y[i + D/2] = x2 (c r) - x1 (s r)
// The result is rounded to bf16 (a quantisation), so the fp32 evaluation is pinned to one fixed
// sequence of correctly rounded operations:
//   - sum of squares in 8 partial sums P_m (m = d mod 8), each accumulated over increasing d
//     with fused multiply-adds starting from 0, combined as
//     ss = ((P0 + P2) + (P4 + P6)) + ((P1 + P3) + (P5 + P7));
//   - ms = ss * (1/D); r = 1 / sqrt(ms + eps) as a rounded square root then a rounded division;
//   - c = cos * r, s = sin * r, y1 = fma(x1, c, x2 * s), y2 = fma(x2, c, x1 * (sin * -r))
//     (x1 * (sin * -r) is exactly -(x1 * s)).
// Pairs of lanes go through the packed fp32x2 instructions; each lane is the same IEEE operation
// as its scalar form, so packing does not change any result.
template <int D>
__device__ __forceinline__ uint64_t bf16x2_to_f2(uint32_t w) {
  return f2_pack(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}

__device__ __forceinline__ uint32_t f2_to_bf16x2(uint64_t v) { return pack_bf16x2(f2_lo(v), f2_hi(v)); }

template <int D>
__device__ __forceinline__ void qk_row_transform_packed(uint32_t (&w)[D / 2], int pos, const float4* rope, int rope_T,
                                                        int use_norm, float eps) {
  float r = 1.0f;
  if (use_norm) {
    uint64_t acc[4] = {0, 0, 0, 0};
#pragma unroll
    for (int g = 0; g < D / 8; ++g)
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint64_t x2 = bf16x2_to_f2<D>(w[4 * g + k]);
        acc[k] = f2_fma(x2, x2, acc[k]);
      }
    const uint64_t e = f2_add(f2_add(acc[0], acc[1]), f2_add(acc[2], acc[3]));
    const float ss = __fadd_rn(f2_lo(e), f2_hi(e));
    const float ms = __fmul_rn(ss, 1.0f / D);
    r = __frcp_rn(__fsqrt_rn(__fadd_rn(ms, eps)));
  }
  constexpr int Q4 = D / 4;  // words per half row
  if (rope != nullptr) {
    const uint64_t r2 = f2_pack(r, r), nr2 = f2_pack(-r, -r);
    const float4* cs = rope + pos;
#pragma unroll
    for (int i2 = 0; i2 < Q4; ++i2) {
      const float4 t = __ldg(cs + static_cast<size_t>(i2) * rope_T);
      const uint64_t cos2 = f2_pack(t.x, t.y), sin2 = f2_pack(t.z, t.w);
      const uint64_t c2 = f2_mul(cos2, r2), s2 = f2_mul(sin2, r2), sn2 = f2_mul(sin2, nr2);
      const uint64_t x1 = bf16x2_to_f2<D>(w[i2]), x2 = bf16x2_to_f2<D>(w[i2 + Q4]);
      const uint64_t y1 = f2_fma(x1, c2, f2_mul(x2, s2));
      const uint64_t y2 = f2_fma(x2, c2, f2_mul(x1, sn2));
      w[i2] = f2_to_bf16x2(y1);
      w[i2 + Q4] = f2_to_bf16x2(y2);
    }
  } else {
    const uint64_t r2 = f2_pack(r, r);
#pragma unroll
    for (int k = 0; k < D / 2; ++k) w[k] = f2_to_bf16x2(f2_mul(bf16x2_to_f2<D>(w[k]), r2));
  }
}

// One row of D bf16 values as D/2 packed words <-> D/8 16-byte chunks.
template <int D>
__device__ __forceinline__ void set_chunk(uint32_t (&w)[D / 2], int ch, uint4 u) {
  w[4 * ch + 0] = u.x;
  w[4 * ch + 1] = u.y;
  w[4 * ch + 2] = u.z;
  w[4 * ch + 3] = u.w;
}
template <int D>
__device__ __forceinline__ uint4 get_chunk(const uint32_t (&w)[D / 2], int ch) {
  return make_uint4(w[4 * ch + 0], w[4 * ch + 1], w[4 * ch + 2], w[4 * ch + 3]);
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
