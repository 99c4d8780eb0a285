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
//      dQ^_i is added to the fp32 workspace with vector reductions; dV_j and dK^_j stay in TMEM to
//      the end, where dK^ goes through the norm and RoPE backward and both are written in fp32;
//   3. dq: the norm and RoPE backward of the accumulated dq^.
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
  float* delta;               // workspace: [B, H, T]
  float* dqh;                 // workspace: dq^ accumulator (unscaled) [B, T, H, D]
  const float4* rope;         // cos/sin table as in AttnParams, or nullptr
  int rope_T;
  int* err;
  int B, H, Hkv, kv_group, T;
  int window, causal, use_norm;
  float eps;
  float scale_log2;  // log2(e) / sqrt(D)
  float scale;       // 1 / sqrt(D)
  int n_ktiles;      // ceil(T / 128)
};

struct BwdMaps {
  CUtensorMap qh, kh, v, dout;  // 128-row tiles of one head, swizzled as the tensor core reads them
};

// ------------------------------------------------------------------------------------------------
// 1. prep

template <int D>
__device__ __forceinline__ void load_row_words(const __nv_bfloat16* src, uint32_t (&w)[D / 2]) {
  const uint4* s4 = reinterpret_cast<const uint4*>(src);
#pragma unroll
  for (int c = 0; c < D / 8; ++c) set_chunk<D>(w, c, __ldg(s4 + c));
}

template <int D>
__global__ void __launch_bounds__(256) attn_bwd_prep_kernel(const BwdParams p) {
  const long long nq = static_cast<long long>(p.B) * p.T * p.H;
  const long long nk = static_cast<long long>(p.B) * p.T * p.Hkv;
  for (long long row = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; row < nq + nk;
       row += static_cast<long long>(gridDim.x) * blockDim.x) {
    const bool isq = row < nq;
    const long long r = isq ? row : row - nq;
    const int heads = isq ? p.H : p.Hkv;
    const int t = static_cast<int>((r / heads) % p.T);
    uint32_t w[D / 2];
    load_row_words<D>((isq ? p.q : p.k) + r * D, w);
    // the forward's prologue arithmetic, operation for operation: the same bf16 q^, k^
    qk_row_transform_packed<D>(w, t, p.rope, p.rope_T, p.use_norm, p.eps);
    uint4* dst = reinterpret_cast<uint4*>((isq ? p.qh : p.kh) + r * D);
#pragma unroll
    for (int c = 0; c < D / 8; ++c) dst[c] = get_chunk<D>(w, c);
    if (isq) {
      const int h = static_cast<int>(r % p.H);
      const long long b = r / (static_cast<long long>(p.T) * p.H);
      const uint4* o4 = reinterpret_cast<const uint4*>(p.out + r * D);
      const uint4* g4 = reinterpret_cast<const uint4*>(p.dout + r * D);
      float acc = 0.f;
#pragma unroll
      for (int c = 0; c < D / 8; ++c) {
        float o[8], g[8];
        bf16x8_to_f32(__ldg(o4 + c), o);
        bf16x8_to_f32(__ldg(g4 + c), g);
#pragma unroll
        for (int e = 0; e < 8; ++e) acc = fmaf(g[e], o[e], acc);
      }
      p.delta[(b * p.H + h) * p.T + t] = acc;
      float4* z = reinterpret_cast<float4*>(p.dqh + r * D);
#pragma unroll
      for (int c = 0; c < D / 4; ++c) z[c] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
}

// ------------------------------------------------------------------------------------------------
// Norm + RoPE backward of one row, in place: dy (fp32, D values, gradient of the rotated and
// normalised row) -> dx, given the raw row x (bf16) at position pos.

template <int D>
__device__ __forceinline__ void prologue_backward_row(float (&g)[D], const __nv_bfloat16* xrow, int pos,
                                                      const BwdParams& p) {
  constexpr int H2 = D / 2;
  uint32_t w[D / 2];  // the raw row, bf16 pairs (element 2k in the low half of w[k])
  load_row_words<D>(xrow, w);
  auto elem = [&](int d) {
    return __uint_as_float((d & 1) ? (w[d >> 1] & 0xFFFF0000u) : (w[d >> 1] << 16));
  };
  const float4* tab = p.rope != nullptr ? p.rope + pos : nullptr;
  // rotated (unnormalised) pair i: rx1 = x1 c + x2 s, rx2 = x2 c - x1 s; the table holds pairs 2m, 2m + 1
  auto rotated = [&](int i, float cs, float sn, float& r1, float& r2) {
    const float x1 = elem(i), x2 = elem(i + H2);
    if (tab != nullptr) {
      r1 = fmaf(x1, cs, x2 * sn);
      r2 = fmaf(x2, cs, -(x1 * sn));
    } else {
      r1 = x1;
      r2 = x2;
    }
  };
  float r = 1.f, c3 = 0.f;
  if (p.use_norm) {
    float ss = 0.f, dot = 0.f;
#pragma unroll
    for (int m = 0; m < D / 4; ++m) {
      const float4 t = tab != nullptr ? __ldg(tab + static_cast<size_t>(m) * p.rope_T) : make_float4(1.f, 1.f, 0.f, 0.f);
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int i = 2 * m + e;
        float r1, r2;
        rotated(i, e ? t.y : t.x, e ? t.w : t.z, r1, r2);
        ss = fmaf(r1, r1, fmaf(r2, r2, ss));
        dot = fmaf(r1, g[i], fmaf(r2, g[i + H2], dot));
      }
    }
    r = 1.0f / sqrtf(ss * (1.0f / D) + p.eps);
    c3 = r * r * r * (1.0f / D) * dot;
  }
#pragma unroll
  for (int m = 0; m < D / 4; ++m) {
    const float4 t = tab != nullptr ? __ldg(tab + static_cast<size_t>(m) * p.rope_T) : make_float4(1.f, 1.f, 0.f, 0.f);
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int i = 2 * m + e;
      const float cs = e ? t.y : t.x, sn = e ? t.w : t.z;
      float g1 = g[i], g2 = g[i + H2];
      if (p.use_norm) {
        float r1, r2;
        rotated(i, cs, sn, r1, r2);
        g1 = fmaf(r, g1, -(c3 * r1));
        g2 = fmaf(r, g2, -(c3 * r2));
      }
      if (tab != nullptr) {
        g[i] = fmaf(g1, cs, -(g2 * sn));
        g[i + H2] = fmaf(g1, sn, g2 * cs);
      } else {
        g[i] = g1;
        g[i + H2] = g2;
      }
    }
  }
}

// ------------------------------------------------------------------------------------------------
// 3. dq = norm/RoPE backward of dq^ / sqrt(D), one thread per (b, t, h) row

template <int D>
__global__ void __launch_bounds__(128) attn_bwd_dq_kernel(const BwdParams p) {
  const long long nq = static_cast<long long>(p.B) * p.T * p.H;
  for (long long r = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; r < nq;
       r += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int t = static_cast<int>((r / p.H) % p.T);
    float g[D];
    const float4* a4 = reinterpret_cast<const float4*>(p.dqh + r * D);
#pragma unroll
    for (int c = 0; c < D / 4; ++c) {
      const float4 u = a4[c];
      g[4 * c] = u.x * p.scale;
      g[4 * c + 1] = u.y * p.scale;
      g[4 * c + 2] = u.z * p.scale;
      g[4 * c + 3] = u.w * p.scale;
    }
    prologue_backward_row<D>(g, p.q + r * D, t, p);
    float4* o4 = reinterpret_cast<float4*>(p.dq + r * D);
#pragma unroll
    for (int c = 0; c < D / 4; ++c) o4[c] = make_float4(g[4 * c], g[4 * c + 1], g[4 * c + 2], g[4 * c + 3]);
  }
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
      s_delta[s * 128 + tid] = i < p.T ? __ldg(p.delta + o) : 0.f;
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
      prologue_backward_row<D>(g, p.k + row * D, j, p);
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
