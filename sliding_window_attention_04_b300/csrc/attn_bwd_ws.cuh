// Warp-specialised, persistent attention backward main kernel (D = 32, 64): the computation of
// attn_bwd_kernel (attn_bwd.cuh) with the tensor pipe kept busy while the exponentials run and the
// per-tile set-up and write-out hidden behind the next tile.
//
// Work unit (tile): one (batch row, K/V head, 128-key tile j), handed out by a ticket counter in
// the workspace (cleared by the prologue pass) in the order b, K/V head, j: concurrent CTAs work on
// neighbouring key tiles of one head, whose Q^ / dO tiles they share in L2. 16 warps:
//   warp 0      producer: takes tickets and publishes them (two-slot tile ring); K^_j, V_j per tile
//               into a two-slot K/V buffer; per iteration (query head, 128-query tile i) the Q^_i,
//               dO_i tiles by TMA and -lse log2(e), delta of the tile's queries by bulk copies (from
//               the prologue pass's padded rows) into the Q ring;
//   warp 1      MMA issuer (one thread; also allocates TMEM);
//   warps 4-7   softmax A: the first 64 queries of every query tile;  warps 8-11 softmax B: the last 64;
//   warps 12-15 dQ: reads dQ^_i (lane = query row) from TMEM, stages it in shared memory and adds it
//               to the fp32 workspace with TMA reductions; after a tile's last iteration, reads its
//               dV_j and dK^_j from TMEM (releasing the accumulators to the next tile) and stores dv
//               and dk^ / sqrt(D) by TMA (the finalize pass applies the norm and RoPE backward to dk).
// Iterations N are numbered across the CTA's tiles. Iteration N is split into two 64-query halves
// h = 2N (A) and 2N + 1 (B). Half h uses TMEM half-buffer h mod 3 (128 columns: S^T fp32 at +0,
// dP^T fp32 at +64; after its softmax P^T bf16 at +32 and dS^T bf16 at +96) and shared-memory dS^T
// slot h mod 4 (128 keys x 64 queries, bf16, 128-byte swizzle). The issuer runs, for step N:
//   S^T, dP^T of halves (N, A), (N, B)                       -> sdp_full[buffer]
//   dV, dK^ += P^T dO, dS^T Q^ over the queries of (N-1, B) (P^T, dS^T from TMEM); dQ^ = dS K^ for
//   all of N-1 (dS from shared memory), written into the dP^T columns of (N-1, B)'s buffer after the
//   dK^ product before it has read its dS^T there           -> q_empty, dq_full
//   (N-1 the last iteration of its tile: that tile's K/V slot is released and its accumulators
//   handed to the dQ warps -> kv_free, final; the next tile's first dV, dK^ product waits for them
//   to be read -> acc_free)
//   dV, dK^ += ... over the queries of (N, A)                 -> buf_free[(N, A)'s buffer]
// dV and dK^ accumulate in TMEM columns 384 and 384 + D.
//
// Ordering. All tcgen05.mma of the CTA are issued by one thread and execute in issue order, so a
// product that overwrites TMEM or shared memory an earlier product reads needs no barrier. The
// waits that remain: a half-buffer whose previous occupant was a B half also held that
// iteration's dQ^, and is reused only after the dQ warps have read it (buf_free); the dS^T slot of
// half h is rewritten by half h + 4, whose softmax starts after S^T of h + 4, i.e. after the
// products of iteration N(h) + 1 (in issue order) have completed. Every barrier's waiter is at
// most one phase behind (two-slot p_full because softmax B may finish half (N+1, B) before the
// issuer has consumed (N, B); two-slot dq_full because the CTA's last dQ^ product follows the one
// before it with no S^T of a next iteration in between, so both can complete while the dQ warps are
// still writing out the previous tile); every wait is bounded and gives up with the error word set.
#pragma once
#include "attn_bwd.cuh"

namespace swa {

template <int D>
struct BwdWsCfg {
  static_assert(D == 32 || D == 64, "the warp-specialised backward covers D = 32 and 64");
  static constexpr int kThreads = 512;
  static constexpr int kStages = D == 64 ? 2 : 3;  // Q ring (Q^, dO tiles, -lse log2 e, delta)
  static constexpr int kTileBytes = kTile * D * 2;
  static constexpr int kHalfStage = kTile * 64 * 2;  // one dS^T slot: 128 keys x 64 queries
  static constexpr int kOffK = 0;                                // [2] K^ slots
  static constexpr int kOffV = kOffK + 2 * kTileBytes;           // [2] V slots
  static constexpr int kOffQ = kOffV + 2 * kTileBytes;
  static constexpr int kOffDO = kOffQ + kStages * kTileBytes;
  static constexpr int kOffDS = kOffDO + kStages * kTileBytes;  // 4 slots
  static constexpr int kOffStg = kOffDS + 4 * kHalfStage;       // dQ^ / dV / dK staging: 128 rows x 32 fp32
  static constexpr int kOffLse = kOffStg + kTile * 128;         // [kStages][128] -lse log2(e)
  static constexpr int kOffDelta = kOffLse + kStages * 512;     // [kStages][128]
  static constexpr int kOffBar = kOffDelta + kStages * 512;
  // barriers
  static constexpr int kBarTileFull = 0;                 // [2] ticket ring
  static constexpr int kBarTileEmpty = 2;                // [2]
  static constexpr int kBarKVFull = 4;                   // [2]
  static constexpr int kBarKVFree = 6;                   // [2]
  static constexpr int kBarQFull = 8;                    // [kStages]
  static constexpr int kBarQEmpty = kBarQFull + kStages;
  static constexpr int kBarSdp = kBarQEmpty + kStages;   // [3] S^T, dP^T of a half in the buffer
  static constexpr int kBarBufFree = kBarSdp + 3;        // [3]
  static constexpr int kBarPFull = kBarBufFree + 3;      // [2 halves][2 slots]
  static constexpr int kBarDq = kBarPFull + 4;          // [2] dQ^ of iteration N in its buffer (slot N & 1)
  static constexpr int kBarFinal = kBarDq + 2;           // [2] a tile's accumulators complete
  static constexpr int kBarAccFree = kBarFinal + 2;      // the accumulators have been read
  static constexpr int kNumBars = kBarAccFree + 1;
  static constexpr int kTileConsumers = 1 + 8 + 1;      // issuer, softmax warps, dQ warpgroup
  static constexpr int kOffMisc = kOffBar + 8 * kNumBars;  // tmem address, abort flag, tile ids [2], dQ-warps flag
  static constexpr int kSmemBytes = kOffMisc + 32 + 1024;
  static constexpr uint32_t kColDV = 384;
  static constexpr uint32_t kColDK = 384 + D;
  static constexpr uint32_t kTmemCols = 512;
  static __host__ __device__ constexpr uint32_t col_buf(int buf) { return 128u * buf; }
};

// Fetch a tensor-map box into L2 only (no shared memory, no completion to wait for).
__device__ __forceinline__ void tma_prefetch_l2_4d(const void* tmap, int x, int y, int z, int w) {
  asm volatile("cp.async.bulk.prefetch.tensor.4d.L2.global.tile [%0, {%1, %2, %3, %4}];" ::"l"(
                   reinterpret_cast<uint64_t>(tmap)),
               "r"(x), "r"(y), "r"(z), "r"(w)
               : "memory");
}

// One work tile: (batch row b, K/V head hk, key tile jt) and the query tiles it meets.
struct BwdTile {
  int b, hk, j0, it_lo, n_it, n_iter;
  __device__ __forceinline__ void set(const BwdParams& p, int t) {
    const int jt = t % p.n_ktiles;
    const int bh = t / p.n_ktiles;
    hk = bh % p.Hkv;
    b = bh / p.Hkv;
    j0 = jt * kTile;
    int hi;
    query_tile_range(p, j0, it_lo, hi);
    n_it = hi - it_lo + 1;  // >= 1: the tile's own query tile always sees it
    n_iter = n_it * p.kv_group;
  }
  // iteration n of the tile: query head hk * kv_group + n / n_it, query tile it_lo + n % n_it
  __device__ __forceinline__ int head(const BwdParams& p, int n) const { return hk * p.kv_group + n / n_it; }
  __device__ __forceinline__ int q0(int n) const { return (it_lo + n % n_it) * kTile; }
};

__device__ __forceinline__ void named_barrier(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// Bits c (0..31) with lo <= c <= hi.
__device__ __forceinline__ uint32_t vis_bits(int lo, int hi) {
  const uint32_t upper = hi >= 31 ? 0xFFFFFFFFu : (hi < 0 ? 0u : (0xFFFFFFFFu >> (31 - hi)));
  const uint32_t lower = lo <= 0 ? 0xFFFFFFFFu : (lo > 31 ? 0u : (0xFFFFFFFFu << lo));
  return upper & lower;
}

// The queries that see key j form one interval [lo, hi] (empty when lo > hi).
__device__ __forceinline__ void visible_queries(const BwdParams& p, int j, int& lo, int& hi) {
  if (j >= p.T) {
    lo = 1;
    hi = 0;
    return;
  }
  lo = p.causal ? j : (p.window >= 0 ? j - p.window : 0);
  hi = p.T - 1;
  if (p.window >= 0 && j + p.window < hi) hi = j + p.window;
  if (lo < 0) lo = 0;
}

// One 64-query half of a 128 x 128 score tile for this thread's key row: P^T = exp2(S^T scale -
// lse log2 e) (zero where the query does not see the key) and dS^T = P^T (dP^T - delta), both
// rounded to bf16: P^T into TMEM at +32 of the half-buffer and dS^T at +96 (blocks in the order 1,
// 0, over fp32 columns already read), dS^T also into the shared-memory slot (for dQ^).
__device__ __forceinline__ void bwd_softmax_half(uint32_t tX, const float* nlse, const float* dl, uint8_t* slot,
                                                 int row, bool masked, int vlo, int vhi, uint64_t scale2) {
#pragma unroll 1
  for (int k = 0; k < 2; ++k) {
    const int blk = 1 - k;
    uint32_t sv[32], pv[32];
    __syncwarp();
    tmem_ld32(tX + 32 * blk, sv);
    tmem_ld32(tX + 64 + 32 * blk, pv);
    tmem_ld_wait();
    reg_fence<32>(sv);
    reg_fence<32>(pv);
    const uint32_t vis = masked ? vis_bits(vlo - 32 * blk, vhi - 32 * blk) : 0xFFFFFFFFu;
    uint32_t pw[16], dw[16];
#pragma unroll
    for (int c = 0; c < 32; c += 4) {
      const float4 nl = *reinterpret_cast<const float4*>(nlse + 32 * blk + c);
      const float4 de = *reinterpret_cast<const float4*>(dl + 32 * blk + c);
#pragma unroll
      for (int e = 0; e < 4; e += 2) {
        const uint64_t s2 = f2_pack(__uint_as_float(sv[c + e]), __uint_as_float(sv[c + e + 1]));
        const uint64_t x2 = f2_fma(s2, scale2, e == 0 ? f2_pack(nl.x, nl.y) : f2_pack(nl.z, nl.w));
        float p0 = ex2_approx(f2_lo(x2)), p1 = ex2_approx(f2_hi(x2));
        if (!((vis >> (c + e)) & 1u)) p0 = 0.f;
        if (!((vis >> (c + e + 1)) & 1u)) p1 = 0.f;
        const uint64_t p2 = f2_pack(p0, p1);
        const uint64_t dp2 = f2_pack(__uint_as_float(pv[c + e]), __uint_as_float(pv[c + e + 1]));
        const uint64_t nd2 = e == 0 ? f2_pack(-de.x, -de.y) : f2_pack(-de.z, -de.w);
        const uint64_t ds2 = f2_mul(p2, f2_add(dp2, nd2));
        pw[(c + e) >> 1] = f2_to_bf16x2(p2);
        dw[(c + e) >> 1] = f2_to_bf16x2(ds2);
      }
    }
    tmem_st16(tX + 32 + 16 * blk, pw);
    tmem_st16(tX + 96 + 16 * blk, dw);
    // dS^T row: queries 32 blk .. +31 are 16-byte units 4 blk .. 4 blk + 3 of the 128-byte row
    uint8_t* rowp = slot + row * 128;
#pragma unroll
    for (int u = 0; u < 4; ++u)
      *reinterpret_cast<uint4*>(rowp + (((4 * blk + u) ^ (row & 7)) << 4)) =
          make_uint4(dw[4 * u], dw[4 * u + 1], dw[4 * u + 2], dw[4 * u + 3]);
  }
}

template <int D>
__global__ void __launch_bounds__(512, 1)
    attn_bwd_ws_kernel(const BwdParams p, const __grid_constant__ BwdMaps maps, int* tickets, int n_tiles) {
  using Cfg = BwdWsCfg<D>;
  using G = TileGeom<D>;
  constexpr int S = Cfg::kStages;
  constexpr int TB = Cfg::kTileBytes;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Cfg::kOffBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Cfg::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Cfg::kOffMisc + 4);
  volatile int* tile_id = reinterpret_cast<volatile int*>(smem + Cfg::kOffMisc + 8);  // [2]
  auto bar = [&](int i) { return bars + i; };
  float* s_nlse = reinterpret_cast<float*>(smem + Cfg::kOffLse);
  float* s_delta = reinterpret_cast<float*>(smem + Cfg::kOffDelta);
  uint8_t* stg = smem + Cfg::kOffStg;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(Cfg::kBarTileFull + i), 1);
      mbar_init(bar(Cfg::kBarTileEmpty + i), Cfg::kTileConsumers);
      mbar_init(bar(Cfg::kBarKVFull + i), 1);
      mbar_init(bar(Cfg::kBarKVFree + i), 1);
      mbar_init(bar(Cfg::kBarFinal + i), 1);
    }
    for (int s = 0; s < S; ++s) {
      mbar_init(bar(Cfg::kBarQFull + s), 1);
      mbar_init(bar(Cfg::kBarQEmpty + s), 1);
    }
    for (int i = 0; i < 3; ++i) {
      mbar_init(bar(Cfg::kBarSdp + i), 1);
      mbar_init(bar(Cfg::kBarBufFree + i), 1);
    }
    for (int i = 0; i < 4; ++i) mbar_init(bar(Cfg::kBarPFull + i), 4);
    mbar_init(bar(Cfg::kBarDq), 1);
    mbar_init(bar(Cfg::kBarDq + 1), 1);
    mbar_init(bar(Cfg::kBarAccFree), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
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
  auto wait = [&](int i, uint32_t parity) { return mbar_wait_or_abort(bar(i), parity, abort_flag); };
  // the next tile of the ticket ring (tl-th of this CTA); -1 when none is left, -2 on timeout.
  // The issuer and every softmax warp arrive once on the slot's empty barrier after reading it (the dQ
  // warpgroup reads it through its leader).
  auto next_tile = [&](int tl, bool one_thread) -> int {
    const int slot = tl & 1;
    int t = -1;
    if (one_thread || lane == 0) {
      t = wait(Cfg::kBarTileFull + slot, (tl >> 1) & 1) ? tile_id[slot] : -2;
      mbar_arrive(bar(Cfg::kBarTileEmpty + slot));
    }
    if (!one_thread) t = __shfl_sync(0xffffffffu, t, 0);
    return t;
  };

  if (warp == 0) {
    // ---------------- producer ----------------
    if (lane == 0) {
      bool ok = true;
      prefetch_tmap(&maps.qh);
      prefetch_tmap(&maps.kh);
      prefetch_tmap(&maps.v);
      prefetch_tmap(&maps.dout);
      int N = 0;
      for (int tl = 0; ok; ++tl) {
        const int slot = tl & 1;
        if (tl >= 2 && !wait(Cfg::kBarTileEmpty + slot, ((tl >> 1) - 1) & 1)) {
          ok = false;
          break;
        }
        int t = atomicAdd(tickets, 1);
        if (t >= n_tiles) t = -1;
        tile_id[slot] = t;
        mbar_arrive(bar(Cfg::kBarTileFull + slot));
        if (t < 0) break;
        BwdTile w;
        w.set(p, t);
        if (tl >= 2 && !wait(Cfg::kBarKVFree + slot, ((tl >> 1) - 1) & 1)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(bar(Cfg::kBarKVFull + slot), 2 * TB);
        tma_load_4d(smem + Cfg::kOffK + slot * TB, &maps.kh, bar(Cfg::kBarKVFull + slot), 0, w.hk, w.j0, w.b);
        tma_load_4d(smem + Cfg::kOffV + slot * TB, &maps.v, bar(Cfg::kBarKVFull + slot), 0, w.hk, w.j0, w.b);
        for (int n = 0; n < w.n_iter; ++n, ++N) {
          const int s = N % S;
          const int h = w.head(p, n), i0 = w.q0(n);
          if (N >= S && !wait(Cfg::kBarQEmpty + s, ((N / S) & 1) ^ 1)) {
            ok = false;
            break;
          }
          uint64_t* full = bar(Cfg::kBarQFull + s);
          mbar_arrive_expect_tx(full, 2 * TB + 1024);
          tma_load_4d(smem + Cfg::kOffQ + s * TB, &maps.qh, full, 0, h, i0, w.b);
          tma_load_4d(smem + Cfg::kOffDO + s * TB, &maps.dout, full, 0, h, i0, w.b);
          const size_t o = (static_cast<size_t>(w.b) * p.H + h) * p.Tp + i0;
          bulk_load_1d(s_nlse + s * 128, p.nlse + o, 512, full);
          bulk_load_1d(s_delta + s * 128, p.delta + o, 512, full);
          // warm L2 for the iteration whose stage this one frees next (the load itself waits for it)
          if (n + S < w.n_iter) {
            tma_prefetch_l2_4d(&maps.qh, 0, w.head(p, n + S), w.q0(n + S), w.b);
            tma_prefetch_l2_4d(&maps.dout, 0, w.head(p, n + S), w.q0(n + S), w.b);
          }
        }
      }
      if (!ok) fail();
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer ----------------
      constexpr uint32_t idesc_s = make_idesc_bf16(128, 64, false);            // S^T / dP^T halves: N = 64
      constexpr uint32_t idesc_o = make_idesc_bf16(128, D, true);              // dV, dK^: B MN-major
      constexpr uint32_t idesc_q = make_idesc_bf16(128, D, true) | (1u << 15);  // dQ^: A and B MN-major
      const uint32_t sDS = smem_u32(smem + Cfg::kOffDS);
      bool ok = true;
      // dV += P^T dO and dK^ += dS^T Q^ over the 64 queries of half h (Q ring stage s)
      auto dvdk = [&](int h, int s, bool start) {
        const int half = h & 1;
        const uint32_t pa = tmem + Cfg::col_buf(h % 3) + 32;
        const uint32_t sQ = smem_u32(smem + Cfg::kOffQ + s * TB), sDO = smem_u32(smem + Cfg::kOffDO + s * TB);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const int ks = 4 * half + kk;  // 16 queries per step
          const uint64_t ob = make_sdesc(sDO + ks * 16 * G::kRowBytes, 16, G::kSBO, G::kSwizzle);
          umma_ts(tmem + Cfg::kColDV, pa + kk * 8, ob, idesc_o, start && kk == 0 ? 0u : 1u);
        }
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const int ks = 4 * half + kk;
          // dS^T from TMEM (its half-buffer's dP^T columns), Q^ as the MN-major B
          const uint64_t qb = make_sdesc(sQ + ks * 16 * G::kRowBytes, 16, G::kSBO, G::kSwizzle);
          umma_ts(tmem + Cfg::kColDK, pa + 64 + kk * 8, qb, idesc_o, start && kk == 0 ? 0u : 1u);
        }
      };
      // the B half and dQ^ of iteration m (K/V slot kvs); if it closes tile tl, release that tile
      auto finish = [&](int m, int kvs, bool closes, int tl) -> bool {
        const int s = m % S, h = 2 * m + 1;
        if (!wait(Cfg::kBarPFull + 2 + (m & 1), (m >> 1) & 1)) return false;
        tc_fence_after();
        dvdk(h, s, false);
        const uint32_t pair = sDS + ((2 * m) & 3) * Cfg::kHalfStage;  // the iteration's two dS^T slots, adjacent
        const uint32_t sK = smem_u32(smem + Cfg::kOffK + kvs * TB);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          const uint64_t da = make_sdesc(pair + ks * 16 * 128, Cfg::kHalfStage, 1024, 2);
          const uint64_t kb = make_sdesc(sK + ks * 16 * G::kRowBytes, 16, G::kSBO, G::kSwizzle);
          umma_ss(tmem + Cfg::col_buf(h % 3) + 64, da, kb, idesc_q, ks > 0 ? 1u : 0u);
        }
        umma_commit(bar(Cfg::kBarQEmpty + s));
        umma_commit(bar(Cfg::kBarDq + (m & 1)));
        if (closes) {
          umma_commit(bar(Cfg::kBarKVFree + kvs));
          umma_commit(bar(Cfg::kBarFinal + (tl & 1)));
        }
        return true;
      };
      int N = 0;
      int prev_kvs = 0, prev_tl = -1;
      bool prev_closes = false;
      for (int tl = 0; ok; ++tl) {
        const int t = next_tile(tl, true);
        if (t == -2) { ok = false; break; }
        if (t < 0) break;
        BwdTile w;
        w.set(p, t);
        const int kvs = tl & 1;
        if (!wait(Cfg::kBarKVFull + kvs, (tl >> 1) & 1)) { ok = false; break; }
        const uint32_t sK = smem_u32(smem + Cfg::kOffK + kvs * TB), sV = smem_u32(smem + Cfg::kOffV + kvs * TB);
        for (int n = 0; n < w.n_iter && ok; ++n, ++N) {
          const int s = N % S;
          if (!wait(Cfg::kBarQFull + s, (N / S) & 1)) { ok = false; break; }
          const uint32_t sQ = smem_u32(smem + Cfg::kOffQ + s * TB), sDO = smem_u32(smem + Cfg::kOffDO + s * TB);
          for (int half = 0; half < 2 && ok; ++half) {
            const int h = 2 * N + half, buf = h % 3;
            if (h >= 3 && !wait(Cfg::kBarBufFree + buf, ((h / 3) - 1) & 1)) { ok = false; break; }
            tc_fence_after();
            const uint32_t col = tmem + Cfg::col_buf(buf);
#pragma unroll
            for (int ks = 0; ks < G::kKSteps; ++ks) {
              const uint64_t ka = make_sdesc(sK + G::kstep_off(ks), 16, G::kSBO, G::kSwizzle);
              const uint64_t qb = make_sdesc(sQ + half * 64 * G::kRowBytes + G::kstep_off(ks), 16, G::kSBO, G::kSwizzle);
              umma_ss(col, ka, qb, idesc_s, ks > 0 ? 1u : 0u);
            }
#pragma unroll
            for (int ks = 0; ks < G::kKSteps; ++ks) {
              const uint64_t va = make_sdesc(sV + G::kstep_off(ks), 16, G::kSBO, G::kSwizzle);
              const uint64_t ob = make_sdesc(sDO + half * 64 * G::kRowBytes + G::kstep_off(ks), 16, G::kSBO, G::kSwizzle);
              umma_ss(col + 64, va, ob, idesc_s, ks > 0 ? 1u : 0u);
            }
            umma_commit(bar(Cfg::kBarSdp + buf));
          }
          if (!ok) break;
          if (N >= 1 && !finish(N - 1, prev_kvs, prev_closes, prev_tl)) { ok = false; break; }
          // a tile's first dV, dK^ product restarts the accumulators: the previous tile's must have been read
          if (n == 0 && tl >= 1 && !wait(Cfg::kBarAccFree, (tl - 1) & 1)) { ok = false; break; }
          if (!wait(Cfg::kBarPFull + (N & 1), (N >> 1) & 1)) { ok = false; break; }
          tc_fence_after();
          dvdk(2 * N, s, n == 0);
          umma_commit(bar(Cfg::kBarBufFree + (2 * N) % 3));
          prev_kvs = kvs;
          prev_tl = tl;
          prev_closes = n == w.n_iter - 1;
        }
      }
      if (ok && N >= 1 && !finish(N - 1, prev_kvs, prev_closes, prev_tl)) ok = false;
      if (!ok) fail();
    }
  } else if (warp >= 4 && warp < 12) {
    // ---------------- softmax A (warps 4-7) / B (warps 8-11) ----------------
    const int half = warp >= 8 ? 1 : 0;
    const int row = tid & 127;  // key row = TMEM lane
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint64_t scale2 = f2_pack(p.scale_log2, p.scale_log2);
    bool ok = true;
    int N = 0;
    for (int tl = 0; ok; ++tl) {
      const int t = next_tile(tl, false);
      if (t == -2) { ok = false; break; }
      if (t < 0) break;
      BwdTile w;
      w.set(p, t);
      const int j = w.j0 + row;
      int vlo, vhi;
      visible_queries(p, j, vlo, vhi);
      for (int n = 0; n < w.n_iter; ++n, ++N) {
        const int s = N % S, h = 2 * N + half, buf = h % 3;
        if (!wait(Cfg::kBarQFull + s, (N / S) & 1) || !wait(Cfg::kBarSdp + buf, (h / 3) & 1)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const int q0 = w.q0(n) + 64 * half;
        const bool masked = __any_sync(0xffffffffu, q0 + 63 > vhi || q0 < vlo);
        bwd_softmax_half(tmem + lane_base + Cfg::col_buf(buf), s_nlse + s * 128 + 64 * half,
                         s_delta + s * 128 + 64 * half, smem + Cfg::kOffDS + (h & 3) * Cfg::kHalfStage, row, masked,
                         vlo - q0, vhi - q0, scale2);
        tmem_st_wait();
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(Cfg::kBarPFull + 2 * half + (N & 1)));
      }
    }
    if (!ok && lane == 0) fail();
  } else if (warp >= 12) {
    // ---------------- dQ drains and the per-tile write-out of dV, dK^ ----------------
    const int row = tid & 127;  // TMEM lane: query row for dQ^, key row for dV / dK^
    const bool leader = tid == 12 * 32;
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    volatile int* wg_ok = reinterpret_cast<volatile int*>(smem + Cfg::kOffMisc + 16);
    bool ok = true;
    int N = 0;
    volatile int* wg_tile = wg_ok + 1;
    for (int tl = 0; ok; ++tl) {
      if (leader) {
        const int slot = tl & 1;
        *wg_tile = wait(Cfg::kBarTileFull + slot, (tl >> 1) & 1) ? tile_id[slot] : -2;
        mbar_arrive(bar(Cfg::kBarTileEmpty + slot));
      }
      named_barrier(1, 128);
      const int t = *wg_tile;
      if (t == -2) { ok = false; break; }
      if (t < 0) break;
      BwdTile w;
      w.set(p, t);
      for (int n = 0; n < w.n_iter; ++n, ++N) {
        // one thread waits (bounded) and hands the outcome to the others through the warpgroup barrier,
        // so that all four warps leave together on a timeout and no bar.sync is left waiting
        if (leader) *wg_ok = wait(Cfg::kBarDq + (N & 1), (N >> 1) & 1) ? 1 : 0;
        named_barrier(1, 128);
        if (*wg_ok == 0) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t col = tmem + lane_base + Cfg::col_buf((2 * N + 1) % 3) + 64;
        uint32_t a[D / 32][32];
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          __syncwarp();
          tmem_ld32(col + 32 * c, a[c]);
        }
        tmem_ld_wait();
#pragma unroll
        for (int c = 0; c < D / 32; ++c) reg_fence<32>(a[c]);
        // every lane's dQ^ columns have been read: the half-buffer may be reused at once
        tc_fence_before();
        named_barrier(1, 128);
        if (leader) mbar_arrive(bar(Cfg::kBarBufFree + (2 * N + 1) % 3));
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          if (leader) bulk_wait_group_read0();  // the previous bulk operation has read the box
          named_barrier(1, 128);
          stage_row32(stg, row, a[c]);
          fence_proxy_async_smem();
          named_barrier(1, 128);
          if (leader) {
            tma_reduce_add_4d(&maps.dqh, stg, 32 * c, w.head(p, n), w.q0(n), w.b);
            bulk_commit_group();
          }
        }
      }
      if (!ok) break;
      // ---- write-out of the tile's dV and dK^ / sqrt(D) ----
      // dV goes through the dS^T slot pair of the tile's last iteration (its dQ^ product, the slots'
      // last reader, has completed with the accumulators), dK^ through registers; the accumulators
      // are released once both are read and dV's box copies have left the slots (the slots' next
      // writer is a softmax that starts after the next tile's first dV, dK^ product).
      if (leader) *wg_ok = wait(Cfg::kBarFinal + (tl & 1), (tl >> 1) & 1) && *abort_flag == 0 ? 1 : 0;
      named_barrier(1, 128);
      if (*wg_ok == 0) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint8_t* pair = smem + Cfg::kOffDS + ((2 * (N - 1)) & 3) * Cfg::kHalfStage;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t a[32];
        __syncwarp();
        tmem_ld32(tmem + lane_base + Cfg::kColDV + 32 * c, a);
        tmem_ld_wait();
        reg_fence<32>(a);
        stage_row32(pair + c * (kTile * 128), row, a);
      }
      fence_proxy_async_smem();
      named_barrier(1, 128);
      if (leader) {
#pragma unroll
        for (int c = 0; c < D / 32; ++c) tma_store_4d(&maps.dv, pair + c * (kTile * 128), 32 * c, w.hk, w.j0, w.b);
        bulk_commit_group();
      }
      uint32_t dk[D / 32][32];
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        __syncwarp();
        tmem_ld32(tmem + lane_base + Cfg::kColDK + 32 * c, dk[c]);
      }
      tmem_ld_wait();
#pragma unroll
      for (int c = 0; c < D / 32; ++c) reg_fence<32>(dk[c]);
      tc_fence_before();
      if (leader) bulk_wait_group_read0();
      named_barrier(1, 128);
      if (leader) mbar_arrive(bar(Cfg::kBarAccFree));
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
#pragma unroll
        for (int e = 0; e < 32; ++e) dk[c][e] = __float_as_uint(__uint_as_float(dk[c][e]) * p.scale);
        if (c > 0 && leader) bulk_wait_group_read0();
        named_barrier(1, 128);
        stage_row32(stg, row, dk[c]);
        fence_proxy_async_smem();
        named_barrier(1, 128);
        if (leader) {
          tma_store_4d(&maps.dk, stg, 32 * c, w.hk, w.j0, w.b);
          bulk_commit_group();
        }
      }
    }
    if (leader) bulk_wait_group0();
    if (!ok && lane == 0) fail();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, Cfg::kTmemCols);
  }
}

}  // namespace swa
