// Attention backward: dq, dk, dv of sum(out * dout) for the forward of attn_fwd_ws.cuh (QK-norm +
// RoPE prologue, sliding-window softmax(q^ k^T / sqrt(D)) V), consuming the forward's LSE.
//
// The pages train the model: the "Autoresearch" deep dive's train.py calls loss.backward() through
// CausalSelfAttention.forward (apply_rotary_emb, norm, the attention call), whose autocast forward
// hands bf16 q^, k^ to the attention kernel. The gradient is therefore taken at the bf16 q^, k^ and
// passes back through the bf16 cast unchanged, then through the RMSNorm and the rotation:
//   P    = exp(s - lse),  s = q^ . k^ / sqrt(D) on the visible keys
//   dV   = P^T dO,  dP = dO V^T,  delta_i = dO_i . out_i,  dS = P (dP - delta)
//   dq^  = dS k^ / sqrt(D),  dk^ = dS^T q^ / sqrt(D)
//   norm y = x r, r = (mean(x^2) + eps)^(-1/2):  dx = r dy - (r^3 / D) (x . dy) x
//   RoPE rotates each pair (i, i + D/2) by +angle, so its transpose rotates by -angle.
//
// Three kernels:
//   1. prep: q^, k^ (the forward's own fp32 evaluation, rounded to bf16) into the workspace,
//      delta = rowsum(dO * out) in fp32, and the fp32 dq^ accumulator cleared;
//   2. main, one CTA per (batch row, K/V head, 128-key tile j): K^_j, V_j stay in shared memory
//      while the CTA walks every query head of the group and every 128-query tile i that sees a key
//      of the tile. Per (head, i), on the tensor cores (tcgen05, fp32 accumulators in TMEM):
//        S^T  = K^_j Q^_i^T,   dP^T = V_j dO_i^T                  (128 x 128 each, SS)
//      then each thread (one key row) forms P^T = exp2(S^T log2e/sqrt(D) - lse log2e) and
//      dS^T = P^T (dP^T - delta) in fp32, rounds both to bf16 into TMEM (over the fp32 columns it
//      has read) and dS^T also into shared memory, and
//        dV_j += P^T dO_i,  dK^_j += dS^T Q^_i                     (TS: A from TMEM)
//        dQ^_i = dS K^_j                                           (SS: A = dS^T read M-major)
//      dQ^_i is added to the fp32 workspace; dV_j and dK^_j stay in TMEM to the end, where dv and
//      dk^ / sqrt(D) are written in fp32 (attn_bwd_ws.cuh holds the warp-specialised form of this
//      kernel used for D = 32 and 64; this synchronous form serves D = 128);
//   3. finalize: the norm and RoPE backward of dq^ / sqrt(D) and, in place, of dk^ / sqrt(D).
// dk and dv are deterministic; dq sums the key tiles' contributions in the order they arrive.
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>

#include "attn_common.cuh"

namespace swa {

struct BwdParams {
  const __nv_bfloat16* q;     // [B, T, H, D]
  const __nv_bfloat16* k;     // [B, T, Hkv, D]
  const __nv_bfloat16* v;     // [B, T, Hkv, D]
  const __nv_bfloat16* out;   // [B, T, H, D], the forward's output
  const float* lse;           // [B, H, T], natural log
  const __nv_bfloat16* dout;  // [B, T, H, D]
  float* dq;                  // [B, T, H, D]
  float* dk;                  // [B, T, Hkv, D]
  float* dv;                  // [B, T, Hkv, D]
  __nv_bfloat16* qh;          // workspace: q^ [B, T, H, D]
  __nv_bfloat16* kh;          // workspace: k^ [B, T, Hkv, D]
  float* delta;               // workspace: delta = rowsum(dO * out), [B, H, Tp]
  float* nlse;                // workspace: -lse log2(e), [B, H, Tp] (padding: -inf)
  float* dqh;                 // workspace: dq^ accumulator (unscaled) [B, T, H, D]
  int* tickets;               // workspace: work counter of the persistent kernel (cleared by the prologue)
  const float4* rope;         // cos/sin table position-major: entry m of position t at rope[t * D/4 + m]
                              // (cos_2m, cos_2m+1, sin_2m, sin_2m+1), or nullptr
  int* err;
  int B, H, Hkv, kv_group, T;
  int window, causal, use_norm;
  float eps;
  float scale_log2;  // log2(e) / sqrt(D)
  float scale;       // 1 / sqrt(D)
  int n_ktiles;      // ceil(T / 128)
  int Tp;            // n_ktiles * 128: row length of delta / nlse (padded with -inf / 0 past T)
};

struct BwdMaps {
  CUtensorMap qh, kh, v, dout;  // 128-row tiles of one head, swizzled as the tensor core reads them
  CUtensorMap dqh, dk, dv;      // fp32 [B, T, heads, D]: 128 rows x 32 columns per box, 128-byte swizzle
};

// 1-D bulk copy global -> shared (both 16-byte aligned, size a multiple of 16), counted on `bar`.
__device__ __forceinline__ void bulk_load_1d(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_u32(dst)),
               "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}

// Shared -> global element-wise fp32 add of one tensor-map box (rows past the tensor are dropped).
__device__ __forceinline__ void tma_reduce_add_4d(const void* tmap, const void* src, int x, int y, int z, int w) {
  asm volatile(
      "cp.reduce.async.bulk.tensor.4d.global.shared::cta.add.tile.bulk_group [%0, {%2, %3, %4, %5}], [%1];" ::"l"(
          reinterpret_cast<uint64_t>(tmap)),
      "r"(smem_u32(src)), "r"(x), "r"(y), "r"(z), "r"(w)
      : "memory");
}

// 32 fp32 values of row `row` into a 128-row x 32-column box staged with the 128-byte swizzle
// (16-byte unit u of row r at position u ^ (r & 7)).
__device__ __forceinline__ void stage_row32(uint8_t* box, int row, const uint32_t (&a)[32]) {
  uint8_t* rp = box + row * 128;
#pragma unroll
  for (int u = 0; u < 8; ++u)
    *reinterpret_cast<uint4*>(rp + ((u ^ (row & 7)) << 4)) = make_uint4(a[4 * u], a[4 * u + 1], a[4 * u + 2], a[4 * u + 3]);
}

// ------------------------------------------------------------------------------------------------
// 1. prep
//
// Both passes around the main kernel stream rows; with plain loads they were bound by memory latency
// (few bytes in flight per warp). Every warp owns a ring of shared-memory stages and fills them with cp.async (16-byte chunks, each copy instruction
// covering contiguous bytes), kStages - 1 groups of rows ahead of the group it computes, so the
// next group's loads are in flight without being held in registers. A warp touches only its own
// stages: cp.async.wait_group then __syncwarp() publishes a stage to the warp's lanes, and a
// __syncwarp() after the computation ends their reads before the stage is refilled. There is no
// wait on another warp.

template <int D>
struct PrepCfg {
  static constexpr int kWarps = 8;
  static constexpr int kStages = 2;                 // one group in flight while one is computed
  static constexpr int kMinCtas = 2;                // registers for two CTAs (16 warps) per SM; at D = 128
                                                    // shared memory holds one
  static constexpr int kQRows = 16;                 // rows of a q group: q, out, dout and lse
  static constexpr int kKRows = 48;                 // rows of a k group (the same bytes per stage)
  static constexpr int kArr = kQRows * 2 * D;       // 16 bf16 rows
  static constexpr int kStageBytes = 3 * kArr + kQRows * 4;
  static constexpr int kSmemBytes = kWarps * kStages * kStageBytes;
};

// Byte offset of 16-byte chunk c of staged bf16 row r. Rows are 2D bytes apart and the chunk index
// is XOR-swizzled per row, so that the two-lanes-per-row reads below (16 rows, 8 bytes per lane)
// take the minimum two shared-memory wavefronts.
template <int D>
__device__ __forceinline__ uint32_t prep_pos(int r, int c) {
  const int sw = D == 32 ? ((r >> 1) & 3) : (r & 7);
  return static_cast<uint32_t>(r * 2 * D + 16 * (c ^ sw));
}

// Fill one stage with group `grp` (q groups first, then k groups) and commit it; past the last group
// the commit is empty, which keeps one commit per iteration.
template <int D>
__device__ __forceinline__ void prep_issue(const BwdParams& p, uint8_t* sb, uint32_t grp, uint32_t nqg, uint32_t nkg,
                                           uint32_t nq, uint32_t nk, int lane) {
  using C = PrepCfg<D>;
  constexpr int NC = D / 8;
  if (grp < nqg) {
    const uint32_t row0 = grp * C::kQRows;
    for (int i = lane; i < C::kQRows * NC; i += 32) {
      const int r = i / NC, c = i % NC;
      const uint32_t row = row0 + r;
      const bool v = row < nq;
      const size_t off = static_cast<size_t>(v ? row : 0) * D + 8 * c;
      const uint32_t pos = prep_pos<D>(r, c), n = v ? 16u : 0u;
      cp_async16(sb + pos, p.q + off, n);
      cp_async16(sb + C::kArr + pos, p.out + off, n);
      cp_async16(sb + 2 * C::kArr + pos, p.dout + off, n);
    }
    if (lane < C::kQRows) {
      const uint32_t row = row0 + lane;
      if (row < nq) {
        const uint32_t bt = row / static_cast<uint32_t>(p.H);
        const uint32_t h = row - bt * p.H, t = bt % static_cast<uint32_t>(p.T), b = bt / static_cast<uint32_t>(p.T);
        cp_async4(sb + 3 * C::kArr + 4 * lane, p.lse + (static_cast<size_t>(b) * p.H + h) * p.T + t);
      }
    }
  } else if (grp < nqg + nkg) {
    const uint32_t row0 = (grp - nqg) * C::kKRows;
    for (int i = lane; i < C::kKRows * NC; i += 32) {
      const int r = i / NC, c = i % NC;
      const uint32_t row = row0 + r;
      const bool v = row < nk;
      cp_async16(sb + prep_pos<D>(r, c), p.k + static_cast<size_t>(v ? row : 0) * D + 8 * c, v ? 16u : 0u);
    }
  }
  cp_async_commit();
}

// QK-norm + RoPE of one staged row, two lanes per row as the forward's prologue splits a row: lane e
// owns, in every 16-byte chunk c, the 8 bytes at 8e (elements 8c + 4e .. 8c + 4e + 3). A RoPE pair
// (i, i + D/2) keeps i mod 8, so both elements of a pair belong to one lane; the eight partial sums
// of squares P_m (m = d mod 8) run over the chunks in increasing order, four per lane, and combine
// with one shuffle in the tree ((P0 + P2) + (P4 + P6), (P1 + P3) + (P5 + P7)) of the forward's
// qk_row_transform_packed, so q^ and k^ are bit-identical to the forward's. Every lane of the warp
// calls it (the shuffle); `valid` gates the store.
template <int D>
__device__ __forceinline__ void prep_row(const BwdParams& p, const uint8_t* rows, int rr, int e, bool valid, int t,
                                         __nv_bfloat16* dst_row) {
  constexpr int NC = D / 8;
  uint64_t x[2 * NC];  // x[2c], x[2c + 1]: elements 8c + 4e + {0, 1} and {2, 3}
#pragma unroll
  for (int c = 0; c < NC; ++c) {
    const uint2 u = *reinterpret_cast<const uint2*>(rows + prep_pos<D>(rr, c) + 8 * e);
    x[2 * c] = bf16x2_to_f2<D>(u.x);
    x[2 * c + 1] = bf16x2_to_f2<D>(u.y);
  }
  float rs = 1.0f;
  if (p.use_norm) {
    uint64_t acc0 = 0, acc1 = 0;  // (P_4e, P_4e+1), (P_4e+2, P_4e+3)
#pragma unroll
    for (int c = 0; c < NC; ++c) {
      acc0 = f2_fma(x[2 * c], x[2 * c], acc0);
      acc1 = f2_fma(x[2 * c + 1], x[2 * c + 1], acc1);
    }
    const uint64_t mine = f2_add(acc0, acc1);  // e=0: (P0+P2, P1+P3); e=1: (P4+P6, P5+P7)
    const uint64_t other = __shfl_xor_sync(0xffffffffu, mine, 1);
    const uint64_t tot = e == 0 ? f2_add(mine, other) : f2_add(other, mine);
    const float ss = __fadd_rn(f2_lo(tot), f2_hi(tot));
    const float ms = __fmul_rn(ss, 1.0f / D);
    rs = __frcp_rn(__fsqrt_rn(__fadd_rn(ms, p.eps)));
  }
  const uint64_t r2 = f2_pack(rs, rs);
  uint2* dst = reinterpret_cast<uint2*>(dst_row) + e;
  if (p.rope != nullptr) {
    const uint64_t nr2 = f2_pack(-rs, -rs);
    const float4* tab = p.rope + static_cast<size_t>(t) * (D / 4);
#pragma unroll
    for (int c = 0; c < NC / 2; ++c) {
      uint32_t wa[2], wb[2];
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        // pairs 8c + 4e + 2q + {0, 1}: table entry 4c + 2e + q
        const float4 tt = __ldg(tab + 4 * c + 2 * e + q);
        const uint64_t cos2 = f2_pack(tt.x, tt.y), sin2 = f2_pack(tt.z, tt.w);
        const uint64_t c2 = f2_mul(cos2, r2), s2 = f2_mul(sin2, r2), sn2 = f2_mul(sin2, nr2);
        const uint64_t x1 = x[2 * c + q], x2 = x[2 * (c + NC / 2) + q];
        wa[q] = f2_to_bf16x2(f2_fma(x1, c2, f2_mul(x2, s2)));
        wb[q] = f2_to_bf16x2(f2_fma(x2, c2, f2_mul(x1, sn2)));
      }
      if (valid) {
        dst[2 * c] = make_uint2(wa[0], wa[1]);
        dst[2 * (c + NC / 2)] = make_uint2(wb[0], wb[1]);
      }
    }
  } else {
#pragma unroll
    for (int c = 0; c < NC; ++c)
      if (valid) dst[2 * c] = make_uint2(f2_to_bf16x2(f2_mul(x[2 * c], r2)), f2_to_bf16x2(f2_mul(x[2 * c + 1], r2)));
  }
}

// q^, k^ into the workspace; per q row delta = rowsum(dO * out) (fp32, any order) and -lse log2(e)
// into the padded [B, H, Tp] rows; the dq^ accumulator of the q rows cleared; the ticket counter reset.
template <int D>
__global__ void __launch_bounds__(256, PrepCfg<D>::kMinCtas) attn_bwd_prep_kernel(const BwdParams p) {
  using C = PrepCfg<D>;
  constexpr int NC = D / 8;
  extern __shared__ __align__(16) uint8_t prep_smem[];
  if (blockIdx.x == 0 && threadIdx.x == 0) *p.tickets = 0;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int e = lane & 1, rl = lane >> 1;  // this lane's half and row of a 16-row step
  // row and group indices fit 32 bits: the host admits B T H D < 2^31
  const uint32_t nq = static_cast<uint32_t>(p.B) * p.T * p.H, nk = static_cast<uint32_t>(p.B) * p.T * p.Hkv;
  const uint32_t nqg = (nq + C::kQRows - 1) / C::kQRows, nkg = (nk + C::kKRows - 1) / C::kKRows;
  const uint32_t gw = blockIdx.x * C::kWarps + warp, nw = gridDim.x * C::kWarps;
  uint8_t* ring = prep_smem + warp * C::kStages * C::kStageBytes;
#pragma unroll
  for (int s = 0; s < C::kStages - 1; ++s) prep_issue<D>(p, ring + s * C::kStageBytes, gw + s * nw, nqg, nkg, nq, nk, lane);
  int it = 0;
  for (uint32_t grp = gw; grp < nqg + nkg; grp += nw, ++it) {
    prep_issue<D>(p, ring + ((it + C::kStages - 1) % C::kStages) * C::kStageBytes, grp + (C::kStages - 1) * nw, nqg,
                  nkg, nq, nk, lane);
    cp_async_wait<C::kStages - 1>();
    __syncwarp();
    const uint8_t* sb = ring + (it % C::kStages) * C::kStageBytes;
    if (grp < nqg) {
      const uint32_t row0 = grp * C::kQRows, row = row0 + rl;
      const bool valid = row < nq;
      const uint32_t bt = row / static_cast<uint32_t>(p.H);
      const uint32_t t = bt % static_cast<uint32_t>(p.T);
      prep_row<D>(p, sb, rl, e, valid, static_cast<int>(t), p.qh + static_cast<size_t>(valid ? row : 0) * D);
      uint64_t acc = 0;
#pragma unroll
      for (int c = 0; c < NC; ++c) {
        const uint32_t pos = prep_pos<D>(rl, c) + 8 * e;
        const uint2 uo = *reinterpret_cast<const uint2*>(sb + C::kArr + pos);
        const uint2 ug = *reinterpret_cast<const uint2*>(sb + 2 * C::kArr + pos);
        acc = f2_fma(bf16x2_to_f2<D>(ug.x), bf16x2_to_f2<D>(uo.x), acc);
        acc = f2_fma(bf16x2_to_f2<D>(ug.y), bf16x2_to_f2<D>(uo.y), acc);
      }
      float d = f2_lo(acc) + f2_hi(acc);
      d += __shfl_xor_sync(0xffffffffu, d, 1);
      if (valid && e == 0) {
        const uint32_t h = row - bt * p.H, b = bt / static_cast<uint32_t>(p.T);
        const float lse = *reinterpret_cast<const float*>(sb + 3 * C::kArr + 4 * rl);
        const size_t o = (static_cast<size_t>(b) * p.H + h) * p.Tp + t;
        p.delta[o] = d;
        p.nlse[o] = -lse * 1.4426950408889634f;
      }
      // the group's dq^ rows are contiguous: cleared by coalesced 16-byte stores
      float4* z = reinterpret_cast<float4*>(p.dqh + static_cast<size_t>(row0) * D);
      for (int i = lane; i < C::kQRows * D / 4; i += 32)
        if (row0 + i / (D / 4) < nq) z[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    } else {
      const uint32_t row0 = (grp - nqg) * C::kKRows;
#pragma unroll 1
      for (int s = 0; s < C::kKRows / 16; ++s) {
        const int rr = 16 * s + rl;
        const uint32_t row = row0 + rr;
        const bool valid = row < nk;
        const uint32_t t = (row / static_cast<uint32_t>(p.Hkv)) % static_cast<uint32_t>(p.T);
        prep_row<D>(p, sb, rr, e, valid, static_cast<int>(t), p.kh + static_cast<size_t>(valid ? row : 0) * D);
      }
    }
    __syncwarp();
  }
  cp_async_wait<0>();
  // padding of delta / nlse past T
  const int pad = p.Tp - p.T;
  if (pad > 0) {
    const long long n_pad = static_cast<long long>(p.B) * p.H * pad;
    for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n_pad;
         i += static_cast<long long>(gridDim.x) * blockDim.x) {
      const long long o = (i / pad) * p.Tp + p.T + i % pad;
      p.delta[o] = 0.f;
      p.nlse[o] = __int_as_float(0xff800000);
    }
  }
}

// ------------------------------------------------------------------------------------------------
// 3. finalize: the norm and RoPE backward of dq^ / sqrt(D) (q rows, from the accumulator) and of
//    dk^ / sqrt(D) (k rows, in place in dk); rows staged as in the prep pass

template <int D>
struct FinCfg {
  static constexpr int kWarps = 8;
  static constexpr int kStages = 2;              // one group in flight while one is computed
  static constexpr int kMinCtas = 4;             // 32 warps per SM: 3 KB stages, at most 64 registers
  static constexpr int kRows = 512 / D;          // rows of a group (q rows, then k rows): 3 KB per stage
  static constexpr int kGBytes = kRows * 4 * D;  // the fp32 gradient rows
  static constexpr int kXBytes = kRows * 2 * D;  // the bf16 q or k rows
  static constexpr int kStageBytes = kGBytes + kXBytes;
  static constexpr int kSmemBytes = kWarps * kStages * kStageBytes;
};

// Lane c of a row owns the RoPE pairs (i, i + D/2) for i = 4c .. 4c + 3: elements 4c .. 4c + 3 of
// both halves of the row, so the rotation and its transpose need no shuffle. In shared memory an odd
// row (at D = 32: a row with bit 1 set) has its two halves swapped, so that the lanes of the rows one
// 32-lane step covers read their first (second) halves in the minimum number of wavefronts.
template <int D>
__device__ __forceinline__ int fin_swap(int r) {
  return D == 32 ? (r >> 1) & 1 : r & 1;
}
// 16-byte unit u (elements 4u .. 4u + 3) of staged fp32 row r
template <int D>
__device__ __forceinline__ uint32_t fin_gpos(int r, int u) {
  return static_cast<uint32_t>(r * 4 * D + 16 * (u ^ ((r & 1) * (D / 8))));
}
// 8-byte unit j (elements 4j .. 4j + 3) of staged bf16 row r
template <int D>
__device__ __forceinline__ uint32_t fin_xpos(int r, int j) {
  return static_cast<uint32_t>(FinCfg<D>::kGBytes + r * 2 * D + 8 * (j ^ (fin_swap<D>(r) * (D / 8))));
}

template <int D>
__device__ __forceinline__ void fin_issue(const BwdParams& p, uint8_t* sb, uint32_t grp, uint32_t nqg, uint32_t nkg,
                                          uint32_t nq, uint32_t nk, int lane) {
  using C = FinCfg<D>;
  constexpr int NC = D / 8, NU = D / 4;
  if (grp < nqg + nkg) {
    const bool isq = grp < nqg;
    const uint32_t row0 = (isq ? grp : grp - nqg) * C::kRows, n = isq ? nq : nk;
    const float* gsrc = isq ? p.dqh : p.dk;
    const __nv_bfloat16* xsrc = isq ? p.q : p.k;
    for (int i = lane; i < C::kRows * NU; i += 32) {
      const int r = i / NU, u = i % NU;
      const uint32_t row = row0 + r;
      const bool v = row < n;
      cp_async16(sb + fin_gpos<D>(r, u), gsrc + static_cast<size_t>(v ? row : 0) * D + 4 * u, v ? 16u : 0u);
    }
    // 16-byte chunk k of a bf16 row = 8-byte units 2k, 2k + 1 (the swap keeps them adjacent)
    for (int i = lane; i < C::kRows * NC; i += 32) {
      const int r = i / NC, k = i % NC;
      const uint32_t row = row0 + r;
      const bool v = row < n;
      cp_async16(sb + fin_xpos<D>(r, 2 * k), xsrc + static_cast<size_t>(v ? row : 0) * D + 8 * k, v ? 16u : 0u);
    }
  }
  cp_async_commit();
}

// NC = D/8 lanes per row, RPW rows per 32-lane step; the row sums by shuffles among a row's lanes.
template <int D>
__global__ void __launch_bounds__(256, FinCfg<D>::kMinCtas) attn_bwd_dq_kernel(const BwdParams p) {
  using C = FinCfg<D>;
  constexpr int NC = D / 8, RPW = 32 / NC;
  extern __shared__ __align__(16) uint8_t fin_smem[];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int c = lane % NC, sub = lane / NC;
  const uint32_t nq = static_cast<uint32_t>(p.B) * p.T * p.H, nk = static_cast<uint32_t>(p.B) * p.T * p.Hkv;
  const uint32_t nqg = (nq + C::kRows - 1) / C::kRows, nkg = (nk + C::kRows - 1) / C::kRows;
  const uint32_t gw = blockIdx.x * C::kWarps + warp, nw = gridDim.x * C::kWarps;
  uint8_t* ring = fin_smem + warp * C::kStages * C::kStageBytes;
#pragma unroll
  for (int s = 0; s < C::kStages - 1; ++s) fin_issue<D>(p, ring + s * C::kStageBytes, gw + s * nw, nqg, nkg, nq, nk, lane);
  int it = 0;
  for (uint32_t grp = gw; grp < nqg + nkg; grp += nw, ++it) {
    fin_issue<D>(p, ring + ((it + C::kStages - 1) % C::kStages) * C::kStageBytes, grp + (C::kStages - 1) * nw, nqg, nkg,
                 nq, nk, lane);
    cp_async_wait<C::kStages - 1>();
    __syncwarp();
    const uint8_t* sb = ring + (it % C::kStages) * C::kStageBytes;
    const bool isq = grp < nqg;
    const uint32_t row0 = (isq ? grp : grp - nqg) * C::kRows, n = isq ? nq : nk;
    float* gdst = isq ? p.dq : p.dk;
    const float gscale = isq ? p.scale : 1.0f;  // dk^ arrives already divided by sqrt(D)
    const uint32_t heads = static_cast<uint32_t>(isq ? p.H : p.Hkv);
#pragma unroll 1
    for (int s = 0; s < C::kRows / RPW; ++s) {
      const int rr = s * RPW + sub;
      const uint32_t row = row0 + rr;
      const bool valid = row < n;
      const int t = static_cast<int>((row / heads) % static_cast<uint32_t>(p.T));
      // g1, x1: elements 4c .. 4c + 3; g2, x2: elements D/2 + 4c .. D/2 + 4c + 3
      float g1[4], g2[4], x1[4], x2[4];
      {
        const float4 a = *reinterpret_cast<const float4*>(sb + fin_gpos<D>(rr, c));
        const float4 b = *reinterpret_cast<const float4*>(sb + fin_gpos<D>(rr, c + NC));
        g1[0] = a.x * gscale; g1[1] = a.y * gscale; g1[2] = a.z * gscale; g1[3] = a.w * gscale;
        g2[0] = b.x * gscale; g2[1] = b.y * gscale; g2[2] = b.z * gscale; g2[3] = b.w * gscale;
        const uint2 xa = *reinterpret_cast<const uint2*>(sb + fin_xpos<D>(rr, c));
        const uint2 xb = *reinterpret_cast<const uint2*>(sb + fin_xpos<D>(rr, c + NC));
        x1[0] = __uint_as_float(xa.x << 16); x1[1] = __uint_as_float(xa.x & 0xFFFF0000u);
        x1[2] = __uint_as_float(xa.y << 16); x1[3] = __uint_as_float(xa.y & 0xFFFF0000u);
        x2[0] = __uint_as_float(xb.x << 16); x2[1] = __uint_as_float(xb.x & 0xFFFF0000u);
        x2[2] = __uint_as_float(xb.y << 16); x2[3] = __uint_as_float(xb.y & 0xFFFF0000u);
      }
      float cs[4], sn[4];
      if (p.rope != nullptr) {
        // table entry m holds the cos, sin of pairs 2m, 2m + 1: pairs 4c .. 4c + 3 are entries 2c, 2c + 1
        const float4* tab = p.rope + static_cast<size_t>(t) * (D / 4);
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          const float4 tt = __ldg(tab + 2 * c + k);
          cs[2 * k] = tt.x; cs[2 * k + 1] = tt.y; sn[2 * k] = tt.z; sn[2 * k + 1] = tt.w;
        }
        // x <- RoPE(x): first half x1 c + x2 s, second half x2 c - x1 s
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float y1 = fmaf(x1[k], cs[k], x2[k] * sn[k]);
          const float y2 = fmaf(x2[k], cs[k], -(x1[k] * sn[k]));
          x1[k] = y1;
          x2[k] = y2;
        }
      }
      if (p.use_norm) {
        float ss = 0.f, dot = 0.f;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          ss = fmaf(x1[k], x1[k], ss);
          dot = fmaf(x1[k], g1[k], dot);
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          ss = fmaf(x2[k], x2[k], ss);
          dot = fmaf(x2[k], g2[k], dot);
        }
#pragma unroll
        for (int off = 1; off < NC; off <<= 1) {
          ss += __shfl_xor_sync(0xffffffffu, ss, off);
          dot += __shfl_xor_sync(0xffffffffu, dot, off);
        }
        const float r1 = 1.0f / sqrtf(ss * (1.0f / D) + p.eps);
        const float c3 = r1 * r1 * r1 * (1.0f / D) * dot;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          g1[k] = fmaf(r1, g1[k], -(c3 * x1[k]));
          g2[k] = fmaf(r1, g2[k], -(c3 * x2[k]));
        }
      }
      if (p.rope != nullptr) {
        // transpose of the rotation: dx1 = g1 c - g2 s, dx2 = g1 s + g2 c
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float d1 = fmaf(g1[k], cs[k], -(g2[k] * sn[k]));
          const float d2 = fmaf(g1[k], sn[k], g2[k] * cs[k]);
          g1[k] = d1;
          g2[k] = d2;
        }
      }
      if (valid) {
        float4* o4 = reinterpret_cast<float4*>(gdst + static_cast<size_t>(row) * D);
        o4[c] = make_float4(g1[0], g1[1], g1[2], g1[3]);
        o4[c + NC] = make_float4(g2[0], g2[1], g2[2], g2[3]);
      }
    }
    __syncwarp();
  }
  cp_async_wait<0>();
}

// ------------------------------------------------------------------------------------------------
// 2. main kernel

template <int D>
struct BwdCfg {
  static constexpr int kThreads = 128;
  static constexpr int kStages = D == 128 ? 1 : 2;  // Q^ / dO tile buffers (D = 128: shared memory)
  static constexpr int kTileBytes = kTile * D * 2;
  static constexpr int kDsBytes = kTile * kTile * 2;  // dS^T staging, 128 x 128 bf16
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kOffK + kTileBytes;
  static constexpr int kOffQ = kOffV + kTileBytes;
  static constexpr int kOffDO = kOffQ + kStages * kTileBytes;
  static constexpr int kOffDS = kOffDO + kStages * kTileBytes;
  static constexpr int kOffLse = kOffDS + kDsBytes;          // [kStages][128] lse * log2(e)
  static constexpr int kOffDelta = kOffLse + kStages * 512;  // [kStages][128]
  static constexpr int kOffBar = kOffDelta + kStages * 512;
  static constexpr int kBarKV = 0, kBarLoad = 1, kBarMma = 1 + kStages, kNumBars = 2 + kStages;
  static constexpr int kOffMisc = kOffBar + 8 * kNumBars;
  // + alignment slack; at least 116 KB so that one CTA runs per SM: each allocates all 512 TMEM columns
  static constexpr int kSmemBytes = kOffMisc + 16 + 1024 > 116 * 1024 ? kOffMisc + 16 + 1024 : 116 * 1024;
  // TMEM columns (lane = key row for S/dP/dV/dK, query row for dQ)
  static constexpr uint32_t kColS = 0;    // S^T fp32; P^T bf16 at +64 after the softmax
  static constexpr uint32_t kColDP = 128; // dP^T fp32; dS^T bf16 at +64
  static constexpr uint32_t kColDV = 256;
  static constexpr uint32_t kColDK = 256 + D;
  // dQ: D <= 64 after dK; D = 128 in two 64-column halves over the fp32 S^T / dP^T columns the
  // softmax has consumed (0..63 and 128..191; P^T and dS^T live at 64..127 and 192..255)
  static constexpr uint32_t kColDQ0 = D <= 64 ? 256 + 2 * D : 0;
  static constexpr uint32_t kColDQ1 = D <= 64 ? 256 + 2 * D + 64 : 128;
  static constexpr uint32_t kTmemCols = 512;
};

// The 128-query tiles whose queries see a key of the 128-key tile starting at j0.
__device__ __forceinline__ void query_tile_range(const BwdParams& p, int j0, int& lo, int& hi) {
  const int n_qt = p.n_ktiles;
  lo = 0;
  hi = n_qt - 1;
  if (p.causal) lo = j0 / kTile;
  if (p.window >= 0) {
    const long long top = static_cast<long long>(j0) + kTile - 1 + p.window;
    if (top / kTile < hi) hi = static_cast<int>(top / kTile);
    if (!p.causal) {
      const int bottom = j0 - p.window;
      if (bottom > 0 && bottom / kTile > lo) lo = bottom / kTile;
    }
  }
}

// Does the score tile (queries from i0, keys from j0) hold an entry that is not visible?
__device__ __forceinline__ bool bwd_tile_needs_mask(const BwdParams& p, int i0, int j0) {
  if (i0 + kTile > p.T || j0 + kTile > p.T) return true;
  if (p.causal && j0 + kTile - 1 > i0) return true;
  if (p.window >= 0) {
    if (j0 < i0 + kTile - 1 - p.window) return true;
    if (!p.causal && j0 + kTile - 1 > i0 + p.window) return true;
  }
  return false;
}

template <int D>
__global__ void __launch_bounds__(128, 1) attn_bwd_kernel(const BwdParams p, const __grid_constant__ BwdMaps maps) {
  using Cfg = BwdCfg<D>;
  using G = TileGeom<D>;
  constexpr int S = Cfg::kStages;
  constexpr int TB = Cfg::kTileBytes;
  constexpr int kBoxes = D > 64 ? D / 64 : 1;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Cfg::kOffBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Cfg::kOffMisc);
  float* s_lse = reinterpret_cast<float*>(smem + Cfg::kOffLse);
  float* s_delta = reinterpret_cast<float*>(smem + Cfg::kOffDelta);
  uint8_t* s_ds = smem + Cfg::kOffDS;

  const int tid = threadIdx.x, warp = tid >> 5;
  const int jt = blockIdx.x % p.n_ktiles;
  const int bh = blockIdx.x / p.n_ktiles;
  const int hk = bh % p.Hkv;
  const int b = bh / p.Hkv;
  const int j0 = jt * kTile;
  int it_lo, it_hi;
  query_tile_range(p, j0, it_lo, it_hi);
  const int n_it = it_hi - it_lo + 1;
  const int n_iter = n_it > 0 ? n_it * p.kv_group : 0;

  if (tid == 0) {
    for (int i = 0; i < Cfg::kNumBars; ++i) mbar_init(bars + i, 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, Cfg::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;

  auto load_tile = [&](uint8_t* dst, const CUtensorMap* map, uint64_t* full, int h, int t) {
#pragma unroll
    for (int x = 0; x < kBoxes; ++x) tma_load_4d(dst + x * kTile * 128, map, full, 64 * x, h, t, b);
  };
  // iteration n: query head h = hk * kv_group + n / n_it, query tile it_lo + n % n_it
  auto issue_load = [&](int n) {
    const int s = n % S;
    const int h = hk * p.kv_group + n / n_it;
    const int i0 = (it_lo + n % n_it) * kTile;
    mbar_arrive_expect_tx(bars + Cfg::kBarLoad + s, 2 * TB);
    load_tile(smem + Cfg::kOffQ + s * TB, &maps.qh, bars + Cfg::kBarLoad + s, h, i0);
    load_tile(smem + Cfg::kOffDO + s * TB, &maps.dout, bars + Cfg::kBarLoad + s, h, i0);
  };

  bool ok = true;
  int issued = 0;  // Q^ / dO loads issued (thread 0)
  int consumed = 0;  // iterations whose loads have landed
  if (tid == 0 && n_iter > 0) {
    prefetch_tmap(&maps.qh);
    prefetch_tmap(&maps.kh);
    prefetch_tmap(&maps.v);
    prefetch_tmap(&maps.dout);
    mbar_arrive_expect_tx(bars + Cfg::kBarKV, 2 * TB);
    load_tile(smem + Cfg::kOffK, &maps.kh, bars + Cfg::kBarKV, hk, j0);
    load_tile(smem + Cfg::kOffV, &maps.v, bars + Cfg::kBarKV, hk, j0);
    for (int n = 0; n < S && n < n_iter; ++n) issue_load(n);
    issued = S < n_iter ? S : n_iter;
  }

  constexpr uint32_t idesc_s = make_idesc_bf16(128, 128, false);
  constexpr uint32_t idesc_o = make_idesc_bf16(128, D, true);
  // dQ^ = dS K^: A (dS^T in shared memory) read MN-major (bit 15), B (K^) MN-major
  constexpr uint32_t idesc_q = make_idesc_bf16(128, D <= 64 ? D : 64, true) | (1u << 15);
  const uint32_t sK = smem_u32(smem + Cfg::kOffK), sV = smem_u32(smem + Cfg::kOffV);
  const uint32_t sDS = smem_u32(s_ds);
  uint32_t mma_phase = 0;
  const int j = j0 + tid;  // this thread's key row (S^T, dP^T, dV, dK lanes)

  for (int n = 0; n < n_iter && ok; ++n) {
    const int s = n % S;
    const int h = hk * p.kv_group + n / n_it;
    const int i0 = (it_lo + n % n_it) * kTile;
    // lse (log2 units) and delta of the tile's queries; queries past T get lse = +inf (P = 0)
    {
      const int i = i0 + tid;
      const size_t o = (static_cast<size_t>(b) * p.H + h) * p.T + i;
      s_lse[s * 128 + tid] = i < p.T ? __ldg(p.lse + o) * 1.4426950408889634f : __int_as_float(0x7f800000);
      s_delta[s * 128 + tid] = i < p.T ? __ldg(p.delta + (static_cast<size_t>(b) * p.H + h) * p.Tp + i) : 0.f;
    }
    if (n == 0 && !mbar_wait(bars + Cfg::kBarKV, 0)) ok = false;
    if (!mbar_wait(bars + Cfg::kBarLoad + s, (n / S) & 1)) ok = false;
    if (!__syncthreads_and(ok)) {
      ok = false;
      break;
    }
    consumed = n + 1;
    const uint32_t sQ = smem_u32(smem + Cfg::kOffQ + s * TB), sDO = smem_u32(smem + Cfg::kOffDO + s * TB);
    if (tid == 0) {
      tc_fence_after();
#pragma unroll
      for (int ks = 0; ks < G::kKSteps; ++ks) {
        const uint64_t ka = make_sdesc(sK + G::kstep_off(ks), 16, G::kSBO, G::kSwizzle);
        const uint64_t qb = make_sdesc(sQ + G::kstep_off(ks), 16, G::kSBO, G::kSwizzle);
        umma_ss(tmem + Cfg::kColS, ka, qb, idesc_s, ks > 0 ? 1u : 0u);
      }
#pragma unroll
      for (int ks = 0; ks < G::kKSteps; ++ks) {
        const uint64_t va = make_sdesc(sV + G::kstep_off(ks), 16, G::kSBO, G::kSwizzle);
        const uint64_t ob = make_sdesc(sDO + G::kstep_off(ks), 16, G::kSBO, G::kSwizzle);
        umma_ss(tmem + Cfg::kColDP, va, ob, idesc_s, ks > 0 ? 1u : 0u);
      }
      umma_commit(bars + Cfg::kBarMma);
    }
    if (!mbar_wait(bars + Cfg::kBarMma, mma_phase & 1)) ok = false;
    ++mma_phase;
    tc_fence_after();

    // ---- P^T and dS^T, one key row per thread, 32 query columns at a time (blocks 3, 2, 0, 1:
    // the bf16 results of block b go to column 64 + 16 b, over fp32 columns already read) ----
    {
      const bool masked = bwd_tile_needs_mask(p, i0, j0);
      const float* lse2 = s_lse + s * 128;
      const float* dl = s_delta + s * 128;
      const uint32_t tS = tmem + lane_base + Cfg::kColS, tP = tmem + lane_base + Cfg::kColDP;
#pragma unroll 1
      for (int bi = 0; bi < 4; ++bi) {
        const int blk = bi == 0 ? 3 : (bi == 1 ? 2 : bi - 2);
        uint32_t sv[32], pv[32];
        __syncwarp();
        tmem_ld32(tS + 32 * blk, sv);
        tmem_ld32(tP + 32 * blk, pv);
        tmem_ld_wait();
        reg_fence<32>(sv);
        reg_fence<32>(pv);
        uint32_t pw[16], dw[16];
#pragma unroll
        for (int c = 0; c < 32; c += 2) {
          float pr[2], ds[2];
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int qc = 32 * blk + c + e;
            float x = ex2_approx(fmaf(__uint_as_float(sv[c + e]), p.scale_log2, -lse2[qc]));
            if (masked && (i0 + qc >= p.T || !key_visible(i0 + qc, j, p.T, p.window, p.causal))) x = 0.f;
            pr[e] = x;
            ds[e] = x * (__uint_as_float(pv[c + e]) - dl[qc]);
          }
          pw[c >> 1] = pack_bf16x2(pr[0], pr[1]);
          dw[c >> 1] = pack_bf16x2(ds[0], ds[1]);
        }
        tmem_st16(tS + 64 + 16 * blk, pw);
        tmem_st16(tP + 64 + 16 * blk, dw);
        // dS^T row `tid`, queries 32 blk .. +31: 64 bytes in the 128-byte-swizzled staging tile
        // (64-query halves 16 KB apart; unit u of row r at position u ^ (r & 7))
        uint8_t* rowp = s_ds + (blk >> 1) * (kTile * 128) + tid * 128;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int unit = (blk & 1) * 4 + u;
          *reinterpret_cast<uint4*>(rowp + ((unit ^ (tid & 7)) << 4)) =
              make_uint4(dw[4 * u], dw[4 * u + 1], dw[4 * u + 2], dw[4 * u + 3]);
        }
      }
      tmem_st_wait();
      fence_proxy_async_smem();
      tc_fence_before();
    }
    if (!__syncthreads_and(ok)) {
      ok = false;
      break;
    }

    if (tid == 0) {
      tc_fence_after();
      const uint32_t first = n == 0 ? 0u : 1u;
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        // dO_i / Q^_i as MN-major B (K = 16 queries per step); P^T, dS^T from TMEM
        const uint64_t ob = make_sdesc(sDO + ks * 16 * G::kRowBytes, D >= 128 ? TB / 2 : 16, G::kSBO, G::kSwizzle);
        umma_ts(tmem + Cfg::kColDV, tmem + Cfg::kColS + 64 + ks * 8, ob, idesc_o, (first || ks > 0) ? 1u : 0u);
      }
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        const uint64_t qb = make_sdesc(sQ + ks * 16 * G::kRowBytes, D >= 128 ? TB / 2 : 16, G::kSBO, G::kSwizzle);
        umma_ts(tmem + Cfg::kColDK, tmem + Cfg::kColDP + 64 + ks * 8, qb, idesc_o, (first || ks > 0) ? 1u : 0u);
      }
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        // dS^T staging as the MN-major A (M = queries in two 64-query halves 16 KB apart, K = 16 keys
        // per step = 2 KB); K^_j as the MN-major B (K = keys)
        const uint64_t da = make_sdesc(sDS + ks * 16 * 128, kTile * 128, 1024, 2);
        if constexpr (D <= 64) {
          const uint64_t kb = make_sdesc(sK + ks * 16 * G::kRowBytes, 16, G::kSBO, G::kSwizzle);
          umma_ss(tmem + Cfg::kColDQ0, da, kb, idesc_q, ks > 0 ? 1u : 0u);
        } else {
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            const uint64_t kb = make_sdesc(sK + half * (TB / 2) + ks * 16 * 128, 16, 1024, 2);
            umma_ss(tmem + (half ? Cfg::kColDQ1 : Cfg::kColDQ0), da, kb, idesc_q, ks > 0 ? 1u : 0u);
          }
        }
      }
      umma_commit(bars + Cfg::kBarMma);
    }
    if (!mbar_wait(bars + Cfg::kBarMma, mma_phase & 1)) ok = false;
    ++mma_phase;
    tc_fence_after();
    // the Q^ / dO stage of this iteration is free: load iteration n + S into it
    if (tid == 0 && ok && n + S < n_iter) {
      issue_load(n + S);
      issued = n + S + 1;
    }

    // ---- dQ^_i partial: one query row per thread, added to the fp32 workspace ----
    {
      const int i = i0 + tid;
      float* dst = p.dqh + ((static_cast<size_t>(b) * p.T + i) * p.H + h) * D;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t a[32];
        const uint32_t col = D <= 64 ? Cfg::kColDQ0 + 32 * c : (c < 2 ? Cfg::kColDQ0 + 32 * c : Cfg::kColDQ1 + 32 * (c - 2));
        __syncwarp();
        tmem_ld32(tmem + lane_base + col, a);
        tmem_ld_wait();
        reg_fence<32>(a);
        if (ok && i < p.T) {
#pragma unroll
          for (int e = 0; e < 32; e += 4)
            asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(dst + 32 * c + e),
                         "f"(__uint_as_float(a[e])), "f"(__uint_as_float(a[e + 1])), "f"(__uint_as_float(a[e + 2])),
                         "f"(__uint_as_float(a[e + 3]))
                         : "memory");
        }
      }
    }
    tc_fence_before();
    if (!__syncthreads_and(ok)) ok = false;
  }

  if (!ok) {
    if (tid == 0) {
      report_error(p.err, kDevErrTimeout);
      // let copies still in flight land before the shared memory is released (bounded waits)
      if (n_iter > 0 && consumed == 0) mbar_wait(bars + Cfg::kBarKV, 0);
      for (int n = consumed; n < issued; ++n) mbar_wait(bars + Cfg::kBarLoad + n % S, (n / S) & 1);
      mbar_wait(bars + Cfg::kBarMma, (mma_phase & 1) ^ 1);
    }
  } else if (n_iter > 0) {
    // ---- epilogue: dV_j and dK_j (through the norm and RoPE backward), one key row per thread ----
    tc_fence_after();
    float g[D];
#pragma unroll
    for (int c = 0; c < D / 32; ++c) {
      uint32_t a[32];
      __syncwarp();
      tmem_ld32(tmem + lane_base + Cfg::kColDV + 32 * c, a);
      tmem_ld_wait();
      reg_fence<32>(a);
#pragma unroll
      for (int e = 0; e < 32; ++e) g[32 * c + e] = __uint_as_float(a[e]);
    }
    const size_t row = (static_cast<size_t>(b) * p.T + j) * p.Hkv + hk;
    if (j < p.T) {
      float4* o4 = reinterpret_cast<float4*>(p.dv + row * D);
#pragma unroll
      for (int c = 0; c < D / 4; ++c) o4[c] = make_float4(g[4 * c], g[4 * c + 1], g[4 * c + 2], g[4 * c + 3]);
    }
#pragma unroll
    for (int c = 0; c < D / 32; ++c) {
      uint32_t a[32];
      __syncwarp();
      tmem_ld32(tmem + lane_base + Cfg::kColDK + 32 * c, a);
      tmem_ld_wait();
      reg_fence<32>(a);
#pragma unroll
      for (int e = 0; e < 32; ++e) g[32 * c + e] = __uint_as_float(a[e]) * p.scale;
    }
    if (j < p.T) {
      float4* o4 = reinterpret_cast<float4*>(p.dk + row * D);
#pragma unroll
      for (int c = 0; c < D / 4; ++c) o4[c] = make_float4(g[4 * c], g[4 * c + 1], g[4 * c + 2], g[4 * c + 3]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, Cfg::kTmemCols);
  }
}

}  // namespace swa
