// Polar Express orthogonalisation (the Muon step of the habr "Autoresearch" deep dive's train.py
// listing, optimiser section): batched bf16 GEMMs on the tensor cores plus the Frobenius
// normalisation.
//
//   X = G / (||G||_F * 1.02 + 1e-6)
//   per step (a, b, c):  wide (rows <= cols): A = X X^T, B = b A + c A A, X = a X + B X
//                        tall (rows > cols):  A = X^T X, B = b A + c A A, X = a X + X B
//
// gemm_kernel<A_MN, B_MN> computes, for every matrix z of a batch,
//   D[z] = alpha * P[z] Q[z] + beta * R[z]      (bf16 in, fp32 accumulation in TMEM, bf16 out)
// with P (M x K) and Q (K x N) read through TMA tensor maps either K-major (rows of K contiguous
// elements) or MN-major (rows of M / N contiguous elements), so X X^T, X^T X, A A and B X all take
// their operands straight from the row-major matrices without a transpose. One 128 x 128 output
// tile per CTA: a TMA producer thread streams 64-deep K slices of P and Q through a 6-stage
// shared-memory ring, one thread issues the tcgen05 MMAs (M = 128, N = 128, K = 16 each), and the
// four warps read the accumulator from TMEM (thread = output row) for the epilogue.
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>

#include "attn_common.cuh"

namespace swa {

struct GemmParams {
  int M, N, K;
  float alpha, beta;
  const __nv_bfloat16* R;  // [batch, M, N] or nullptr (no beta term)
  __nv_bfloat16* D;        // [batch, M, N]
  int* err;
};

struct GemmMaps {
  CUtensorMap p, q;  // 3-D (inner, rows, batch) views; see the host side for the box of each form
};

struct GemmCfg {
  static constexpr int BM = 128, BN = 128, BK = 64, kStages = 6;
  static constexpr int kTileP = BM * BK * 2;  // 16 KB
  static constexpr int kTileQ = BN * BK * 2;  // 16 KB
  static constexpr int kStageBytes = kTileP + kTileQ;
  static constexpr int kOffBar = kStages * kStageBytes;
  static constexpr int kBarFull = 0, kBarEmpty = kStages, kBarDone = 2 * kStages, kNumBars = 2 * kStages + 1;
  static constexpr int kOffMisc = kOffBar + 8 * kNumBars;
  static constexpr int kSmemBytes = kOffMisc + 16 + 1024;
};

// Shared-memory descriptor of K step ks (16 deep) of a 128 x 64 operand tile: K-major (128 rows of
// 128 bytes, 128-byte swizzle) or MN-major (two 64-wide M / N chunks of 64 K rows, 8 KB apart).
template <bool MN>
__device__ __forceinline__ uint64_t gemm_desc(uint32_t tile, int ks) {
  if constexpr (MN) return make_sdesc(tile + ks * 16 * 128, 8192, 1024, 2);
  else return make_sdesc(tile + ks * 32, 16, 1024, 2);
}

template <bool A_MN, bool B_MN>
__global__ void __launch_bounds__(128, 1) gemm_kernel(const GemmParams p, const __grid_constant__ GemmMaps maps) {
  using Cfg = GemmCfg;
  constexpr int S = Cfg::kStages;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Cfg::kOffBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Cfg::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Cfg::kOffMisc + 4);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n0 = blockIdx.x * Cfg::BN, m0 = blockIdx.y * Cfg::BM, z = blockIdx.z;
  const int nk = (p.K + Cfg::BK - 1) / Cfg::BK;

  if (tid == 0) {
    for (int i = 0; i < Cfg::kNumBars; ++i) mbar_init(bars + i, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 128);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  auto stage_p = [&](int s) { return smem + s * Cfg::kStageBytes; };
  auto stage_q = [&](int s) { return smem + s * Cfg::kStageBytes + Cfg::kTileP; };

  if (warp == 0 && lane == 0) {
    // ---- producer: K slices of P and Q ----
    prefetch_tmap(&maps.p);
    prefetch_tmap(&maps.q);
    for (int kt = 0; kt < nk; ++kt) {
      const int s = kt % S, k0 = kt * Cfg::BK;
      if (kt >= S && !mbar_wait_or_abort(bars + Cfg::kBarEmpty + s, ((kt / S) - 1) & 1, abort_flag)) {
        report_error(p.err, kDevErrTimeout);
        *abort_flag = 1;
        break;
      }
      uint64_t* full = bars + Cfg::kBarFull + s;
      mbar_arrive_expect_tx(full, Cfg::kStageBytes);
      if constexpr (A_MN) {
        tma_load_3d(stage_p(s), &maps.p, full, m0, k0, z);
        tma_load_3d(stage_p(s) + 8192, &maps.p, full, m0 + 64, k0, z);
      } else {
        tma_load_3d(stage_p(s), &maps.p, full, k0, m0, z);
      }
      if constexpr (B_MN) {
        tma_load_3d(stage_q(s), &maps.q, full, n0, k0, z);
        tma_load_3d(stage_q(s) + 8192, &maps.q, full, n0 + 64, k0, z);
      } else {
        tma_load_3d(stage_q(s), &maps.q, full, k0, n0, z);
      }
    }
  } else if (warp == 1 && lane == 0) {
    // ---- MMA issuer ----
    constexpr uint32_t idesc = make_idesc_bf16(128, 128, B_MN) | (A_MN ? (1u << 15) : 0u);
    bool ok = true;
    for (int kt = 0; kt < nk; ++kt) {
      const int s = kt % S;
      if (!mbar_wait_or_abort(bars + Cfg::kBarFull + s, (kt / S) & 1, abort_flag)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t sp = smem_u32(stage_p(s)), sq = smem_u32(stage_q(s));
#pragma unroll
      for (int ks = 0; ks < Cfg::BK / 16; ++ks)
        umma_ss(tmem, gemm_desc<A_MN>(sp, ks), gemm_desc<B_MN>(sq, ks), idesc, (kt > 0 || ks > 0) ? 1u : 0u);
      umma_commit(bars + Cfg::kBarEmpty + s);
    }
    if (!ok) {
      report_error(p.err, kDevErrTimeout);
      *abort_flag = 1;
    }
    umma_commit(bars + Cfg::kBarDone);
  }

  // ---- epilogue: thread = output row m0 + tid; 32 columns per TMEM load ----
  const bool ok = mbar_wait_or_abort(bars + Cfg::kBarDone, 0, abort_flag) && *abort_flag == 0;
  tc_fence_after();
  const int row = m0 + tid;
  const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
  const size_t rbase = (static_cast<size_t>(z) * p.M + row) * p.N;
#pragma unroll 1
  for (int c = 0; c < Cfg::BN / 32; ++c) {
    uint32_t a[32];
    __syncwarp();
    tmem_ld32(tmem + lane_base + 32 * c, a);
    tmem_ld_wait();
    reg_fence<32>(a);
    const int nc = n0 + 32 * c;
    if (!ok || row >= p.M || nc >= p.N) continue;
    float r[32];
    const bool full_cols = nc + 32 <= p.N;
    if (p.R != nullptr) {
      if (full_cols) {
        const uint4* r4 = reinterpret_cast<const uint4*>(p.R + rbase + nc);
#pragma unroll
        for (int u = 0; u < 4; ++u) bf16x8_to_f32(__ldg(r4 + u), r + 8 * u);
      } else {
        for (int e = 0; e < 32; ++e) r[e] = nc + e < p.N ? __bfloat162float(p.R[rbase + nc + e]) : 0.f;
      }
    } else {
#pragma unroll
      for (int e = 0; e < 32; ++e) r[e] = 0.f;
    }
    uint32_t o[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      const float d0 = fmaf(p.alpha, __uint_as_float(a[2 * e]), p.beta * r[2 * e]);
      const float d1 = fmaf(p.alpha, __uint_as_float(a[2 * e + 1]), p.beta * r[2 * e + 1]);
      o[e] = pack_bf16x2(d0, d1);
    }
    if (full_cols) {
      uint4* d4 = reinterpret_cast<uint4*>(p.D + rbase + nc);
#pragma unroll
      for (int u = 0; u < 4; ++u) d4[u] = make_uint4(o[4 * u], o[4 * u + 1], o[4 * u + 2], o[4 * u + 3]);
    } else {
      const __nv_bfloat16* ob = reinterpret_cast<const __nv_bfloat16*>(o);
      for (int e = 0; e < 32 && nc + e < p.N; ++e) p.D[rbase + nc + e] = ob[e];
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 128);
  }
}

// Frobenius normalisation, one CTA per matrix, as the listing's bf16 tensor operations round:
//   nrm = bf16(sqrt(sum x^2)) (fp32 sum), t = bf16(nrm * 1.02), den = bf16(t + 1e-6), X = bf16(G / den).
__global__ void __launch_bounds__(512) frob_normalize_kernel(const __nv_bfloat16* G, __nv_bfloat16* X, long long mn) {
  __shared__ float part[16];
  __shared__ float s_den;
  const __nv_bfloat16* g = G + blockIdx.x * mn;
  __nv_bfloat16* x = X + blockIdx.x * mn;
  float ss = 0.f;
  for (long long i = threadIdx.x; i < mn; i += blockDim.x) {
    const float v = __bfloat162float(g[i]);
    ss = fmaf(v, v, ss);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
  if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = ss;
  __syncthreads();
  if (threadIdx.x == 0) {
    float t = 0.f;
    for (int w = 0; w < static_cast<int>(blockDim.x >> 5); ++w) t += part[w];
    const float nrm = __bfloat162float(__float2bfloat16_rn(__fsqrt_rn(t)));
    const float t1 = __bfloat162float(__float2bfloat16_rn(__fmul_rn(nrm, 1.02f)));
    s_den = __bfloat162float(__float2bfloat16_rn(__fadd_rn(t1, 1e-6f)));
  }
  __syncthreads();
  const float den = s_den;
  for (long long i = threadIdx.x; i < mn; i += blockDim.x) x[i] = __float2bfloat16_rn(__fdiv_rn(__bfloat162float(g[i]), den));
}

}  // namespace swa
