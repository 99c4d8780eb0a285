// Attention forward, warp-specialised persistent version (D = 32 or 64).
//
// One CTA per SM (512 threads, 1 CTA/SM: ~200 KB shared memory and all 512 TMEM columns). A work
// unit is (b, h, 256-row query block) = two 128-row query tiles that share one stream of
// 128-key K/V tiles. Units are handed out through a global ticket counter in the order
// (b, h)-major, query block descending, so the four blocks of one head run at about the same time
// on different SMs (their K/V tiles are shared through L2) and the cheap blocks come last.
//
// Roles (warp index: role):
//   0-3   softmax of query tile 0   (thread = query row = TMEM lane)
//   4-7   softmax of query tile 1
//   8-11  prologue: QK RMSNorm + RoPE of the Q tiles and of every K tile, in place in shared
//         memory (TMA writes the raw bf16 rows already in the tensor core's swizzled layout)
//   12    producer: ticket fetch, TMA loads of Q, K, V (lane 0)
//   13    MMA issuer (lane 0) and TMEM owner
//   14-15 idle
//
// TMEM (512 columns): S_t (128 fp32 columns each), P_t (128 bf16 = 64 columns each, not aliased
// with S so that S_t of the next key tile can be computed while P_t is still being consumed),
// O_t (D fp32 columns each).
//
// Per key tile j the MMA issuer runs one tile ahead on S:  S_0(j+1), S_1(j+1), then
// O_0 += P_0(j) V(j), O_1 += P_1(j) V(j). The softmax warps read S_t(j), hand the S columns back,
// compute P_t(j) = exp2(s*scale*log2e - m) with a lazily updated running max m (O and l are
// rescaled only when the tile max exceeds m by more than kRescaleLog2), and write P_t(j) to TMEM.
// At the end of a unit they normalise O_t, stage it as bf16 in the (now free) Q tile buffer and
// store it with one TMA store, and write the per-row log-sum-exp.
//
// Every wait is bounded (kWaitTimeoutNs); a role that gives up records the error, sets a CTA
// abort flag that makes the other roles leave their loops, and the CTA drains its own TMA loads
// and MMAs before freeing TMEM.
#pragma once
#include <cuda.h>

#include "attn_common.cuh"

namespace swa {

template <int D>
struct WsCfg {
  using G = TileGeom<D>;
  static constexpr int kThreads = 512;
  static constexpr int kStages = 4;                      // K/V ring depth
  static constexpr int kTileBytes = G::kBytes;           // one 128 x D bf16 tile
  static constexpr int kOffQ = 0;                        // [2 slots][2 tiles] Q^ / output staging
  static constexpr int kOffK = kOffQ + 4 * kTileBytes;   // [kStages] K^ (transformed in place)
  static constexpr int kOffV = kOffK + kStages * kTileBytes;
  static constexpr int kOffBar = kOffV + kStages * kTileBytes;
  // barrier indices
  static constexpr int kBarQFull = 0;                    // [2] TMA -> prologue
  static constexpr int kBarQReady = 2;                   // [2] prologue -> MMA
  static constexpr int kBarQEmpty = 4;                   // [2] epilogue stores read -> producer
  static constexpr int kBarUnit = 6;                     // [2] producer -> MMA, softmax (unit id)
  static constexpr int kBarKFull = 8;                    // [kStages] TMA -> prologue
  static constexpr int kBarKReady = kBarKFull + kStages; // [kStages] prologue -> MMA
  static constexpr int kBarVFull = kBarKReady + kStages; // [kStages] TMA -> MMA
  static constexpr int kBarKVEmpty = kBarVFull + kStages;// [kStages] MMA commit -> producer
  static constexpr int kBarSFull = kBarKVEmpty + kStages;// [2] MMA commit -> softmax t
  static constexpr int kBarSFree = kBarSFull + 2;        // [2] softmax t read S -> MMA
  static constexpr int kBarPFull = kBarSFree + 2;        // [2] softmax t wrote P -> MMA
  static constexpr int kBarPVDone = kBarPFull + 2;       // [2] MMA commit -> softmax t
  static constexpr int kBarFinal = kBarPVDone + 2;       // MMA drain at exit
  static constexpr int kNumBars = kBarFinal + 1;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;  // tmem slot, abort flag, unit ids
  static constexpr int kSmemBytes = kOffMisc + 64 + 1024;  // + alignment slack
  // TMEM columns
  static constexpr uint32_t kTmemCols = 512;
  static __device__ __forceinline__ uint32_t col_s(int t) { return static_cast<uint32_t>(128 * t); }
  static __device__ __forceinline__ uint32_t col_p(int t) { return static_cast<uint32_t>(256 + 64 * t); }
  static __device__ __forceinline__ uint32_t col_o(int t) { return static_cast<uint32_t>(384 + D * t); }
  static_assert(384 + 2 * D <= 512, "TMEM budget");
  static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
};

constexpr float kRescaleLog2 = 8.0f;  // lazy rescale threshold (log2 units): P stays <= 256

// Geometry of one work unit: two 128-row query tiles starting at qs[t] and the key-tile range
// [kb[t], ke[t]] each needs (empty when kb > ke); [kb_all, ke_all] is their union.
struct UnitGeom {
  int b, h;
  int qs[2];
  int kb[2], ke[2];
  int kb_all, ke_all;
};

__device__ __forceinline__ void unit_geom(const AttnParams& p, int n_qb, int unit, UnitGeom& g) {
  const int bh = unit / n_qb;
  const int qb = n_qb - 1 - (unit - bh * n_qb);
  g.b = bh / p.H;
  g.h = bh - g.b * p.H;
  const int T = p.T;
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    const int qs = qb * 256 + 128 * t;
    g.qs[t] = qs;
    if (qs < T) {
      const int qe = min(T - 1, qs + kTile - 1);
      const int lo = p.window >= 0 ? max(0, qs - p.window) : 0;
      const int hi = p.causal ? qe : (p.window >= 0 ? min(T - 1, qe + p.window) : T - 1);
      g.kb[t] = lo / kTile;
      g.ke[t] = hi / kTile;
    } else {
      g.kb[t] = 1;
      g.ke[t] = 0;
    }
  }
  g.kb_all = g.kb[0];
  g.ke_all = g.kb[1] <= g.ke[1] ? max(g.ke[0], g.ke[1]) : g.ke[0];
  if (g.kb[1] <= g.ke[1]) g.kb_all = min(g.kb_all, g.kb[1]);
}

// Does the 128 x 128 score tile (query rows from qs, keys from k0) contain a masked entry?
__device__ __forceinline__ bool tile_needs_mask(const AttnParams& p, int qs, int k0) {
  if (k0 + kTile - 1 >= p.T) return true;
  if (p.causal && k0 + kTile - 1 > qs) return true;
  if (p.window >= 0) {
    if (k0 < qs + kTile - 1 - p.window) return true;
    if (!p.causal && k0 + kTile - 1 > qs + p.window) return true;
  }
  return false;
}

// QK-norm + RoPE of row `row` of a swizzled 128-row tile, in place.
template <int D>
__device__ __forceinline__ void transform_row_inplace(uint8_t* tile, int row, int pos, const AttnParams& p) {
  float x[D];
#pragma unroll
  for (int ch = 0; ch < D / 8; ++ch)
    bf16x8_to_f32(*reinterpret_cast<const uint4*>(tile + tile_off<D>(row, ch)), x + ch * 8);
  qk_row_transform<D>(x, pos, p.rope, p.use_norm, p.eps,
                      [&](int ch, uint4 u) { *reinterpret_cast<uint4*>(tile + tile_off<D>(row, ch)) = u; });
}

struct WsMaps {
  CUtensorMap q, k, v, out;  // 4-D (D, H, T, B) views, box (D, 1, 128, 1), swizzled
};

template <int D>
__global__ void __launch_bounds__(512, 1)
    attn_fwd_ws_kernel(const AttnParams p, const __grid_constant__ WsMaps maps, int* sched, int n_units) {
  using Cfg = WsCfg<D>;
  constexpr int TB = Cfg::kTileBytes;
  constexpr int S = Cfg::kStages;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Cfg::kOffBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Cfg::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Cfg::kOffMisc + 4);
  volatile int* unit_id = reinterpret_cast<volatile int*>(smem + Cfg::kOffMisc + 8);  // [2]
  auto bar = [&](int i) { return bars + i; };
  auto q_tile = [&](int slot, int t) { return smem + Cfg::kOffQ + (2 * slot + t) * TB; };
  auto k_tile = [&](int st) { return smem + Cfg::kOffK + st * TB; };
  auto v_tile = [&](int st) { return smem + Cfg::kOffV + st * TB; };

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int n_qb = (p.T + 2 * kTile - 1) / (2 * kTile);

  if (tid == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(Cfg::kBarQFull + i), 1);
      mbar_init(bar(Cfg::kBarQReady + i), 4);
      mbar_init(bar(Cfg::kBarQEmpty + i), 2);
      mbar_init(bar(Cfg::kBarUnit + i), 1);
      mbar_init(bar(Cfg::kBarSFull + i), 1);
      mbar_init(bar(Cfg::kBarSFree + i), 4);
      mbar_init(bar(Cfg::kBarPFull + i), 4);
      mbar_init(bar(Cfg::kBarPVDone + i), 1);
    }
    for (int i = 0; i < S; ++i) {
      mbar_init(bar(Cfg::kBarKFull + i), 1);
      mbar_init(bar(Cfg::kBarKReady + i), 4);
      mbar_init(bar(Cfg::kBarVFull + i), 1);
      mbar_init(bar(Cfg::kBarKVEmpty + i), 1);
    }
    mbar_init(bar(Cfg::kBarFinal), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 13) {
    tmem_alloc(tmem_slot, Cfg::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  auto fail = [&]() {
    report_error(p.err, kDevErrTimeout);
    *abort_flag = 1;
  };

  if (warp >= 12) {
    regs_dec<56>();
    if (warp == 12 && lane == 0) {
      // ---------------- producer: tickets and TMA loads ----------------
      prefetch_tmap(&maps.q);
      prefetch_tmap(&maps.k);
      prefetch_tmap(&maps.v);
      prefetch_tmap(&maps.out);
      const uint64_t pol_stream = policy_evict_first();
      const uint64_t pol_keep = policy_evict_last();
      int q_armed[2] = {-1, -1};  // parity of the last armed, not yet drained phase
      int k_armed[S], v_armed[S];
      for (int i = 0; i < S; ++i) k_armed[i] = v_armed[i] = -1;
      uint32_t kcnt = 0;
      bool ok = true;
      for (uint32_t ul = 0;; ++ul) {
        const int slot = ul & 1;
        const uint32_t uph = (ul >> 1) & 1;
        if (!mbar_wait_or_abort(bar(Cfg::kBarQEmpty + slot), uph ^ 1, abort_flag)) {
          ok = false;
          break;
        }
        int unit = ok ? atomicAdd(sched, 1) : n_units;
        if (unit >= n_units) unit = -1;
        unit_id[slot] = unit;
        mbar_arrive(bar(Cfg::kBarUnit + slot));
        if (unit < 0) {
          mbar_arrive(bar(Cfg::kBarQFull + slot));
          break;
        }
        UnitGeom g;
        unit_geom(p, n_qb, unit, g);
        const bool two = g.kb[1] <= g.ke[1];
        mbar_arrive_expect_tx(bar(Cfg::kBarQFull + slot), (two ? 2 : 1) * TB);
        q_armed[slot] = static_cast<int>(uph);
        tma_load_4d_hint(q_tile(slot, 0), &maps.q, bar(Cfg::kBarQFull + slot), 0, g.h, g.qs[0], g.b, pol_stream);
        if (two)
          tma_load_4d_hint(q_tile(slot, 1), &maps.q, bar(Cfg::kBarQFull + slot), 0, g.h, g.qs[1], g.b,
                           pol_stream);
        for (int j = g.kb_all; j <= g.ke_all; ++j, ++kcnt) {
          const int st = kcnt % S;
          const uint32_t ph = (kcnt / S) & 1;
          if (!mbar_wait_or_abort(bar(Cfg::kBarKVEmpty + st), ph ^ 1, abort_flag)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(bar(Cfg::kBarKFull + st), TB);
          k_armed[st] = static_cast<int>(ph);
          tma_load_4d_hint(k_tile(st), &maps.k, bar(Cfg::kBarKFull + st), 0, g.h, j * kTile, g.b, pol_keep);
          mbar_arrive_expect_tx(bar(Cfg::kBarVFull + st), TB);
          v_armed[st] = static_cast<int>(ph);
          tma_load_4d_hint(v_tile(st), &maps.v, bar(Cfg::kBarVFull + st), 0, g.h, j * kTile, g.b, pol_keep);
        }
        if (!ok) break;
      }
      if (!ok) {
        fail();
        // Drain: every TMA load this thread issued must land before the CTA exits.
        for (int i = 0; i < 2; ++i)
          if (q_armed[i] >= 0) mbar_wait(bar(Cfg::kBarQFull + i), static_cast<uint32_t>(q_armed[i]));
        for (int i = 0; i < S; ++i) {
          if (k_armed[i] >= 0) mbar_wait(bar(Cfg::kBarKFull + i), static_cast<uint32_t>(k_armed[i]));
          if (v_armed[i] >= 0) mbar_wait(bar(Cfg::kBarVFull + i), static_cast<uint32_t>(v_armed[i]));
        }
      }
      // The last CTA to leave resets the ticket counters for the next launch on this slot.
      __threadfence();
      const int done = atomicAdd(sched + 1, 1);
      if (done == static_cast<int>(gridDim.x) - 1) {
        atomicExch(sched, 0);
        atomicExch(sched + 1, 0);
      }
    } else if (warp == 13 && lane == 0) {
      // ---------------- MMA issuer ----------------
      using G = TileGeom<D>;
      constexpr uint32_t idesc_s = make_idesc_bf16(128, 128, false);
      constexpr uint32_t idesc_o = make_idesc_bf16(128, D, true);
      uint32_t kcnt = 0;
      uint32_t scnt[2] = {0, 0}, pcnt[2] = {0, 0};
      bool ok = true;
      for (uint32_t ul = 0; ok; ++ul) {
        const int slot = ul & 1;
        const uint32_t uph = (ul >> 1) & 1;
        if (!mbar_wait_or_abort(bar(Cfg::kBarUnit + slot), uph, abort_flag)) {
          ok = false;
          break;
        }
        const int unit = unit_id[slot];
        if (unit < 0) break;
        if (!mbar_wait_or_abort(bar(Cfg::kBarQReady + slot), uph, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        UnitGeom g;
        unit_geom(p, n_qb, unit, g);
        const uint32_t qa[2] = {smem_u32(q_tile(slot, 0)), smem_u32(q_tile(slot, 1))};

        auto issue_s = [&](int j, uint32_t kc) -> bool {
          const int st = kc % S;
          if (!mbar_wait_or_abort(bar(Cfg::kBarKReady + st), (kc / S) & 1, abort_flag)) return false;
          tc_fence_after();
          const uint32_t ka = smem_u32(k_tile(st));
          for (int t = 0; t < 2; ++t) {
            if (j < g.kb[t] || j > g.ke[t]) continue;
            if (!mbar_wait_or_abort(bar(Cfg::kBarSFree + t), (scnt[t] & 1) ^ 1, abort_flag)) return false;
            tc_fence_after();
#pragma unroll
            for (int ks = 0; ks < G::kKSteps; ++ks) {
              const uint64_t ad = make_sdesc(qa[t] + G::kstep_off(ks), 16, G::kSBO, G::kSwizzle);
              const uint64_t bd = make_sdesc(ka + G::kstep_off(ks), 16, G::kSBO, G::kSwizzle);
              umma_ss(tmem + Cfg::col_s(t), ad, bd, idesc_s, ks > 0 ? 1u : 0u);
            }
            umma_commit(bar(Cfg::kBarSFull + t));
            ++scnt[t];
          }
          return true;
        };
        auto issue_pv = [&](int j, uint32_t kc) -> bool {
          const int st = kc % S;
          if (!mbar_wait_or_abort(bar(Cfg::kBarVFull + st), (kc / S) & 1, abort_flag)) return false;
          tc_fence_after();
          const uint32_t va = smem_u32(v_tile(st));
          for (int t = 0; t < 2; ++t) {
            if (j < g.kb[t] || j > g.ke[t]) continue;
            if (!mbar_wait_or_abort(bar(Cfg::kBarPFull + t), pcnt[t] & 1, abort_flag)) return false;
            tc_fence_after();
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
              const uint64_t bd = make_sdesc(va + ks * 16 * G::kRowBytes, 16, G::kSBO, G::kSwizzle);
              umma_ts(tmem + Cfg::col_o(t), tmem + Cfg::col_p(t) + ks * 8, bd, idesc_o,
                      (j > g.kb[t] || ks > 0) ? 1u : 0u);
            }
            umma_commit(bar(Cfg::kBarPVDone + t));
            ++pcnt[t];
          }
          umma_commit(bar(Cfg::kBarKVEmpty + st));
          return true;
        };

        const uint32_t kc0 = kcnt;
        for (int j = g.kb_all; j <= g.ke_all && ok; ++j) {
          const uint32_t kc = kc0 + static_cast<uint32_t>(j - g.kb_all);
          if (!issue_s(j, kc)) ok = false;
          else if (j > g.kb_all && !issue_pv(j - 1, kc - 1)) ok = false;
        }
        if (ok && !issue_pv(g.ke_all, kc0 + static_cast<uint32_t>(g.ke_all - g.kb_all))) ok = false;
        kcnt = kc0 + static_cast<uint32_t>(g.ke_all - g.kb_all + 1);
      }
      if (!ok) fail();
      // Drain: all MMAs this thread issued complete before TMEM is freed.
      umma_commit(bar(Cfg::kBarFinal));
      mbar_wait(bar(Cfg::kBarFinal), 0);
    }
  } else if (warp >= 8) {
    regs_dec<104>();
    // ---------------- prologue: QK-norm + RoPE in place ----------------
    const int r = tid - 256;  // row of the tile this thread transforms
    uint32_t kcnt = 0;
    bool ok = true;
    for (uint32_t ul = 0;; ++ul) {
      const int slot = ul & 1;
      const uint32_t uph = (ul >> 1) & 1;
      ok = __all_sync(0xffffffffu, mbar_wait_or_abort(bar(Cfg::kBarQFull + slot), uph, abort_flag));
      if (!ok) break;
      const int unit = unit_id[slot];
      if (unit < 0) break;
      UnitGeom g;
      unit_geom(p, n_qb, unit, g);
      for (int t = 0; t < 2; ++t) {
        if (g.kb[t] > g.ke[t]) continue;
        const int pos = g.qs[t] + r;
        transform_row_inplace<D>(q_tile(slot, t), r, pos < p.T ? pos : 0, p);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(Cfg::kBarQReady + slot));
      for (int j = g.kb_all; j <= g.ke_all; ++j, ++kcnt) {
        const int st = kcnt % S;
        ok = __all_sync(0xffffffffu, mbar_wait_or_abort(bar(Cfg::kBarKFull + st), (kcnt / S) & 1, abort_flag));
        if (!ok) break;
        const int pos = j * kTile + r;
        transform_row_inplace<D>(k_tile(st), r, pos < p.T ? pos : 0, p);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(Cfg::kBarKReady + st));
      }
      if (!ok) break;
    }
    if (!ok && lane == 0) fail();
  } else {
    regs_inc<176>();
    // ---------------- softmax + epilogue of query tile t ----------------
    const int t = warp >> 2;
    const int r = tid & 127;                                  // row in the tile = TMEM lane
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_base + Cfg::col_s(t);
    const uint32_t tP = tmem + lane_base + Cfg::col_p(t);
    const uint32_t tO = tmem + lane_base + Cfg::col_o(t);
    const float scale = p.scale_log2;
    uint32_t n = 0;  // P tiles written so far by this warpgroup (all units)
    bool ok = true;
    for (uint32_t ul = 0; ok; ++ul) {
      const int slot = ul & 1;
      const uint32_t uph = (ul >> 1) & 1;
      ok = __all_sync(0xffffffffu, mbar_wait_or_abort(bar(Cfg::kBarUnit + slot), uph, abort_flag));
      if (!ok) break;
      const int unit = unit_id[slot];
      if (unit < 0) break;
      UnitGeom g;
      unit_geom(p, n_qb, unit, g);
      if (g.kb[t] > g.ke[t]) {  // this query tile lies past T
        named_bar_sync(1 + t, 128);
        if (r == 0) mbar_arrive(bar(Cfg::kBarQEmpty + slot));
        continue;
      }
      const int qs = g.qs[t];
      const int i_row = qs + r;
      float m_used = -INFINITY;  // reference max of this row (log2 units)
      float l_run = 0.f;         // sum of exp2(score - m_used)
      for (int j = g.kb[t]; j <= g.ke[t]; ++j, ++n) {
        const int k0 = j * kTile;
        ok = __all_sync(0xffffffffu, mbar_wait_or_abort(bar(Cfg::kBarSFull + t), n & 1, abort_flag));
        if (!ok) break;
        tc_fence_after();
        uint32_t s[128];
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld32(tS + 32 * c, s + 32 * c);
        tmem_ld_wait();
        reg_fence<128>(s);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(Cfg::kBarSFree + t));

        if (tile_needs_mask(p, qs, k0)) {
          // visible columns of this row: lo <= c <= hi
          int lo = p.window >= 0 ? i_row - p.window - k0 : -1;
          int hi = p.causal ? i_row - k0 : (p.window >= 0 ? i_row + p.window - k0 : kTile);
          hi = min(hi, p.T - 1 - k0);
#pragma unroll
          for (int c = 0; c < 128; ++c)
            if (c < lo || c > hi) s[c] = __float_as_uint(-INFINITY);
        }
        float mx0 = -INFINITY, mx1 = -INFINITY, mx2 = -INFINITY, mx3 = -INFINITY;
#pragma unroll
        for (int c = 0; c < 128; c += 8) {
          mx0 = fmax3(mx0, __uint_as_float(s[c + 0]), __uint_as_float(s[c + 1]));
          mx1 = fmax3(mx1, __uint_as_float(s[c + 2]), __uint_as_float(s[c + 3]));
          mx2 = fmax3(mx2, __uint_as_float(s[c + 4]), __uint_as_float(s[c + 5]));
          mx3 = fmax3(mx3, __uint_as_float(s[c + 6]), __uint_as_float(s[c + 7]));
        }
        const float m_tile = fmax3(mx0, mx1, fmaxf(mx2, mx3)) * scale;
        const bool grow = m_tile > m_used + kRescaleLog2 || (m_used == -INFINITY && m_tile > -INFINITY);
        const float m_new = grow ? m_tile : m_used;
        const float alpha = grow ? ex2_approx(m_used - m_new) : 1.0f;  // 0 when m_used = -inf
        const float m_use = m_new == -INFINITY ? 0.f : m_new;
        const uint64_t scale2 = f2_pack(scale, scale);
        const uint64_t negm2 = f2_pack(-m_use, -m_use);
        uint64_t sum2 = 0;  // two fp32 zeros
        uint32_t pk[64];
#pragma unroll
        for (int c = 0; c < 64; ++c) {
          const uint64_t x2 = f2_fma(f2_pack(__uint_as_float(s[2 * c]), __uint_as_float(s[2 * c + 1])), scale2, negm2);
          const float p0 = ex2_approx(f2_lo(x2));
          const float p1 = ex2_approx(f2_hi(x2));
          const uint64_t pp = f2_pack(p0, p1);
          sum2 = f2_add(sum2, pp);
          pk[c] = pack_bf16x2(p0, p1);
        }
        const float rowsum = f2_lo(sum2) + f2_hi(sum2);

        // P_t(j-1) must have been consumed (and O_t updated) before P and O are touched again.
        if (n > 0) {
          ok = __all_sync(0xffffffffu, mbar_wait_or_abort(bar(Cfg::kBarPVDone + t), (n - 1) & 1, abort_flag));
          if (!ok) break;
          tc_fence_after();
        }
        if (j > g.kb[t] && __any_sync(0xffffffffu, alpha != 1.0f)) {
          uint32_t o[D];
#pragma unroll
          for (int c = 0; c < D / 32; ++c) tmem_ld32(tO + 32 * c, o + 32 * c);
          tmem_ld_wait();
          reg_fence<D>(o);
#pragma unroll
          for (int c = 0; c < D; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * alpha);
#pragma unroll
          for (int c = 0; c < D / 32; ++c) tmem_st32(tO + 32 * c, o + 32 * c);
        }
        l_run = l_run * alpha + rowsum;
        m_used = m_new;
        tmem_st32(tP, pk);
        tmem_st32(tP + 32, pk + 32);
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(Cfg::kBarPFull + t));
      }
      if (!ok) break;
      // ---- epilogue: O / l -> bf16 staged in this tile's Q buffer, one TMA store; LSE ----
      ok = __all_sync(0xffffffffu, mbar_wait_or_abort(bar(Cfg::kBarPVDone + t), (n - 1) & 1, abort_flag));
      if (!ok) break;
      tc_fence_after();
      uint32_t o[D];
#pragma unroll
      for (int c = 0; c < D / 32; ++c) tmem_ld32(tO + 32 * c, o + 32 * c);
      tmem_ld_wait();
      reg_fence<D>(o);
      const float inv_l = l_run > 0.f ? 1.0f / l_run : 0.f;
      uint8_t* stage = q_tile(slot, t);
#pragma unroll
      for (int ch = 0; ch < D / 8; ++ch) {
        uint4 u;
        u.x = pack_bf16x2(__uint_as_float(o[ch * 8 + 0]) * inv_l, __uint_as_float(o[ch * 8 + 1]) * inv_l);
        u.y = pack_bf16x2(__uint_as_float(o[ch * 8 + 2]) * inv_l, __uint_as_float(o[ch * 8 + 3]) * inv_l);
        u.z = pack_bf16x2(__uint_as_float(o[ch * 8 + 4]) * inv_l, __uint_as_float(o[ch * 8 + 5]) * inv_l);
        u.w = pack_bf16x2(__uint_as_float(o[ch * 8 + 6]) * inv_l, __uint_as_float(o[ch * 8 + 7]) * inv_l);
        *reinterpret_cast<uint4*>(stage + tile_off<D>(r, ch)) = u;
      }
      if (p.lse != nullptr && i_row < p.T) {
        const float m_fin = m_used == -INFINITY ? 0.f : m_used;
        p.lse[(static_cast<size_t>(g.b) * p.H + g.h) * p.T + i_row] = (m_fin + __log2f(l_run)) * 0.69314718055994531f;
      }
      fence_proxy_async_smem();
      named_bar_sync(1 + t, 128);
      if (r == 0) {
        tma_store_4d(&maps.out, stage, 0, g.h, qs, g.b);
        bulk_commit_group();
        bulk_wait_group_read0();
        mbar_arrive(bar(Cfg::kBarQEmpty + slot));
      }
    }
    if (!ok && lane == 0) fail();
    if (r == 0) bulk_wait_group0();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 13) {
    tc_fence_after();
    tmem_dealloc(tmem, Cfg::kTmemCols);
  }
}

}  // namespace swa
