// Attention forward, warp-specialised persistent version (D = 32, 64, 128).
//
// One CTA per SM (640 threads = five warpgroups, up to ~200 KB shared memory, all 512 TMEM columns).
// A work unit is (b, h, 256-row query block) = two 128-row query tiles sharing one stream of 128-key
// K/V tiles. A ticket counter hands out chunks of one head's units, run back to back and sharing key
// tiles through the ring: all of a head's blocks where consecutive blocks share tiles (all but the
// last heads), else pairs (blocks qb, qb - 1), heaviest first, so the cheap blocks end the queue.
//
// Roles (warp index: role):
//   0-3    softmax of query tile 0   (thread = query row = TMEM lane)
//   4-7    softmax of query tile 1
//   8-15   prologue: QK RMSNorm + RoPE of the Q tiles and of every K tile, two threads per row,
//          in place in shared memory (TMA writes the raw bf16 rows already in the tensor core's
//          swizzled layout); a row is widened to fp32 once and its cos/sin entries are loaded
//          while its sum of squares is formed
//   16     producer: ticket fetch, TMA loads of Q, K, V (lane 0)
//   17     S issuer (lane 0): S = Q^ K^^T jobs in stream order; TMEM owner
//   18, 19 P.V issuers of query tiles 0 and 1 (lane 0): O_t += P V in order
//
// TMEM (512 columns): kSBufs rotating 128-column S/P buffers (three; two at D = 128) and O_0, O_1
// (D columns each). The S jobs (one per query tile and key tile, in stream order) take the buffers
// round-robin. A softmax warpgroup reads S from its buffer and writes P (bf16, 64 columns) into the
// buffer's upper half once that half has been read, so P needs no space of its own; the P.V MMA
// reads P from there, and its completion frees the buffer for the S job kSBufs places later. With
// three buffers for two query tiles (D <= 64) the S of a tile's next key tile is normally computed
// while its softmax still works on the current one.
//
// Three single-thread MMA issuers each run a plain in-order loop of blocking waits: the S issuer and
// one P.V issuer per query tile, which wakes as soon as its tile's P is written, so one tile's softmax
// never holds up the other tile's MMAs. (Measured: the tensor pipe accepts a new tcgen05.mma only
// about every 64 cycles, so a thread that issues stays blocked while its MMAs run; one thread issuing
// every MMA spends those cycles serially with all of its waits and was slower than three.)
//
// Every wait on a phase-parity barrier is exact: the waiter is never two phases away from the
// barrier. S-done, P-written and P.V-done have two slots per tile, used by the tile's even and odd
// jobs, and S job n of a tile is issued only after the tile's P.V job n - 2 has completed: that P.V
// needed P of job n - 2, so the S-done and P-written slots of job n - 2 have been consumed before
// job n can complete or its P be written, and a softmax that waits for P.V job n - 1 (O rescale,
// epilogue) knows that job n - 3 has completed. Buffer-free is per buffer and waited only by the S
// issuer, which issues the buffer's next S only after the P.V that read it. A softmax writes the P of
// its next job while the previous P.V may still run (the two sit in different buffers); only the O
// rescale and the epilogue wait for that P.V. (tests/test_pipeline_model.py runs every role's waits
// and arrivals under random interleavings and checks these claims.)
//
// Softmax of one S tile. With the QK-norm on (softmax_tile_fixed) every scaled score is bounded, so
// the exponentials use a fixed reference and need no maximum and no rescale. Otherwise (softmax_tile)
// the row max over the four 32-column blocks comes first (reducing TMEM loads), then the exponentials
// block by block. A row's block that the mask removes entirely
// gets zero P without exponentials, and only a block that the mask edge cuts is masked element
// by element; tiles without any masked entry skip the mask tests. The running max is updated lazily:
// O and l are rescaled only when the tile max exceeds the current reference by more than
// kRescaleLog2. At the end of a unit the softmax warps normalise O_t and store it as bf16, each
// thread its own row, and write the per-row log-sum-exp. A Q slot is freed as soon as the unit's last
// S job has read its Q^ tiles (and every role has read the slot's unit id and geometry), so the
// producer loads the Q tiles of the unit after next while the current unit still runs.
//
// Registers: the kernel is compiled to 96 per thread (640 x 96 = 61440); at start the warpgroups
// re-divide them with setmaxnreg: softmax 128, prologue 80, producer/MMA group 64, i.e.
// 128 x (128 + 128 + 80 + 80 + 64) = 61440. The host launches the kernel only when the compiled
// count is exactly kLaunchRegs, so the increase can always be satisfied.
//
// Every wait is bounded (kWaitTimeoutNs); a role that gives up records the error, sets a CTA
// abort flag that makes the other roles leave their loops, and the CTA drains its own TMA loads
// and MMAs before freeing TMEM.
#pragma once
#include <cuda.h>

#include "attn_common.cuh"

namespace swa {

// Arrivals that free a Q slot for the unit two ahead: the S issuer's commit after the unit's last S
// job (its Q^ tiles are no longer read), both P.V issuers and the eight softmax warps once they have
// read the slot's unit id and geometry.
constexpr int kQEmptyArrivals = 1 + 2 + 8;

// Rows of the output box one softmax warp stages and stores (its 32 rows of the query tile).
constexpr int kOutRows = 32;

// Byte offset of 16-byte chunk `ch` of row `row` in a staged output box (the tensor map's swizzle:
// 128-byte rows with the 128-byte pattern, 64-byte rows at D = 32 with the 64-byte pattern).
template <int D>
__device__ __forceinline__ uint32_t out_stage_off(int row, int ch) {
  if constexpr (D >= 64) return static_cast<uint32_t>(row * 128 + ((ch ^ (row & 7)) << 4));
  else return static_cast<uint32_t>(row * 64 + ((ch ^ ((row >> 1) & 3)) << 4));
}

template <int D>
struct WsCfg {
  using G = TileGeom<D>;
  static constexpr int kThreads = 640;
  static constexpr int kLaunchRegs = 96;  // per thread at launch; the run-time split adds up to it
  // D = 128: 32 KB tiles and 128-column O accumulators; one Q slot (the next unit's Q is loaded
  // once the current unit's S jobs are done), a 2-stage ring and two S/P buffers fit shared memory
  // and TMEM.
  static constexpr int kQSlots = D == 128 ? 1 : 2;       // units whose Q tiles are resident at once
  static constexpr int kStages = D == 128 ? 2 : 4;       // K/V ring depth
  static constexpr int kSBufs = D == 128 ? 2 : 3;        // S/P buffers in TMEM
  static constexpr int kTileBytes = G::kBytes;           // one 128 x D bf16 tile
  static constexpr int kOffQ = 0;                        // [kQSlots][2 tiles] Q^
  static constexpr int kOffK = kOffQ + 2 * kQSlots * kTileBytes;  // [kStages] K^ (transformed in place)
  static constexpr int kOffV = kOffK + kStages * kTileBytes;
  // output staging: one box of kOutRows rows x min(D, 64) columns per softmax warp
  static constexpr int kOutBytes = kOutRows * (D > 64 ? 64 : D) * 2;
  static constexpr int kOffOut = kOffV + kStages * kTileBytes;
  static constexpr int kOffBar = kOffOut + 8 * kOutBytes;
  // barrier indices
  static constexpr int kBarQFull = 0;                     // [2] TMA -> prologue
  static constexpr int kBarQReady = 2;                    // [2] prologue -> MMA
  static constexpr int kBarQEmpty = 4;                    // [2] slot free (S issuer, P.V issuers, softmax warps) -> producer
  static constexpr int kBarUnit = 6;                      // [2] producer -> MMA, softmax (unit id)
  static constexpr int kBarKFull = 8;                     // [kStages] TMA -> prologue
  static constexpr int kBarKReady = kBarKFull + kStages;  // [kStages] prologue -> S issuer
  static constexpr int kBarVFull = kBarKReady + kStages;  // [kStages] TMA -> P.V issuers
  static constexpr int kBarKFree = kBarVFull + kStages;   // [kStages] S jobs of the step done -> producer
  static constexpr int kBarVFree = kBarKFree + kStages;   // [kStages] both P.V issuers done with V -> producer
  static constexpr int kBarSFull = kBarVFree + kStages;   // [2 tiles][2] S job n of tile t done -> softmax t
  static constexpr int kBarBufFree = kBarSFull + 4;       // [kSBufs] P.V job done -> S issuer
  static constexpr int kBarPFull = kBarBufFree + kSBufs;  // [2 tiles][2] softmax t wrote P of job n -> P.V issuer t
  static constexpr int kBarPVDone = kBarPFull + 4;        // [2 tiles][2] P.V job n of tile t done -> softmax, S issuer
  static constexpr int kBarFinal = kBarPVDone + 4;        // [3] MMA drain at exit (S issuer, P.V issuers)
  static constexpr int kBarVReady = kBarFinal + 3;        // [kStages] gated calls: prologue gated V -> P.V issuers
  static constexpr int kNumBars = kBarVReady + kStages;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;  // tmem slot, abort flag, unit ids, unit geometry
  static constexpr int kSmemBytes = kOffMisc + 128 + 1024;  // + alignment slack
  static_assert(kSmemBytes <= 232448, "shared memory per CTA");
  // TMEM columns
  static constexpr uint32_t kTmemCols = 512;
  static __device__ __forceinline__ uint32_t col_buf(int b) { return static_cast<uint32_t>(128 * b); }
  static __device__ __forceinline__ uint32_t col_o(int t) { return static_cast<uint32_t>(128 * kSBufs + D * t); }
  static_assert(128 * kSBufs + 2 * D <= 512, "TMEM budget");
  static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
};

constexpr float kRescaleLog2 = 8.0f;  // lazy rescale threshold (log2 units): P stays <= 256

// Geometry of one work unit: two 128-row query tiles starting at qs0, qs0 + 128 and the
// key-tile range [kb_t, ke_t] each needs (empty when kb > ke); [kb_all, ke_all] is their union.
struct UnitGeom {
  int b, h, hk, qs0;  // hk: the K/V head of query head h
  int kb0, ke0, kb1, ke1;
  int kb_all, ke_all;
  // Key steps run from ke_all down to kb_all. The first r_in of them reuse K^ / V tiles the
  // previous unit left in the ring; the last r_out are left there for the next unit.
  int r_in, r_out;
  __device__ __forceinline__ int n_steps() const { return ke_all - kb_all + 1; }
  __device__ __forceinline__ bool has(int t, int j) const {
    return t == 0 ? (j >= kb0 && j <= ke0) : (j >= kb1 && j <= ke1);
  }
  __device__ __forceinline__ int kb(int t) const { return t == 0 ? kb0 : kb1; }
  __device__ __forceinline__ int ke(int t) const { return t == 0 ? ke0 : ke1; }
  __device__ __forceinline__ bool valid(int t) const { return kb(t) <= ke(t); }
};

__device__ __forceinline__ void unit_geom(const AttnParams& p, int bh, int qb, UnitGeom& g) {
  g.r_in = g.r_out = 0;
  g.b = bh / p.H;
  g.h = bh - g.b * p.H;
  g.hk = g.h / p.kv_group;
  g.qs0 = qb * 2 * kTile;
  const int T = p.T;
  int kb[2], ke[2];
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    const int qs = g.qs0 + kTile * t;
    if (qs < T) {
      const int qe = min(T - 1, qs + kTile - 1);
      const int lo = p.window >= 0 ? max(0, qs - p.window) : 0;
      const int hi = p.causal ? qe : (p.window >= 0 ? min(T - 1, qe + p.window) : T - 1);
      kb[t] = lo / kTile;
      ke[t] = hi / kTile;
    } else {
      kb[t] = 1;
      ke[t] = 0;
    }
  }
  g.kb0 = kb[0];
  g.ke0 = ke[0];
  g.kb1 = kb[1];
  g.ke1 = ke[1];
  const bool two = kb[1] <= ke[1];
  g.kb_all = two ? min(kb[0], kb[1]) : kb[0];
  g.ke_all = two ? max(ke[0], ke[1]) : ke[0];
}

// Key tiles that unit `a` (query block qb of a head) and the next unit `nb` of the same CTA (block
// qb - 1 of the same head) can share through the ring: with both streaming key tiles downwards, the
// last R tiles `a` loads are the first R that `nb` needs, in the same (first-in, first-out) order,
// where R = nb.ke_all - a.kb_all + 1. They stay resident when R is at most the ring depth.
template <int S>
__device__ __forceinline__ int shared_steps(const UnitGeom& a, const UnitGeom& nb) {
  if (a.b != nb.b || a.h != nb.h || nb.qs0 + 2 * kTile != a.qs0) return 0;
  const int R = nb.ke_all - a.kb_all + 1;
  return (R >= 1 && R <= S && R <= a.n_steps() && R <= nb.n_steps()) ? R : 0;
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

// Half-row QK-norm + RoPE: a row of D values is shared by two threads; half h owns the elements
// d with d mod 8 in [4h, 4h + 4), i.e. 8 bytes of each 16-byte chunk. RoPE pairs (i, i + D/2) have
// the same d mod 8, so every pair stays inside one thread; the 8 partial sums of squares split
// 4 / 4 and are combined with one shuffle in the order qk_row_transform_packed uses.
template <int D>
struct RopeHalf {
  float4 cs[D / 8];  // (cos, cos, sin, sin) of pairs 2 i2, 2 i2 + 1 for this half's i2 values
  __device__ __forceinline__ void load(const AttnParams& p, int pos, int h) {
    if (p.rope == nullptr) return;
    const float4* src = p.rope + pos;
#pragma unroll
    for (int k = 0; k < D / 8; ++k) {
      const int i2 = 4 * (k >> 1) + 2 * h + (k & 1);  // i2 mod 4 in {2h, 2h + 1}
      cs[k] = __ldg(src + static_cast<size_t>(i2) * p.rope_T);
    }
  }
};

// D = 128: the same arithmetic in two passes over shared memory (the row is widened twice), so that
// the fp32 row and the cos/sin entries never need to be live at once: the sum of squares chunk by
// chunk (the same per-residue order as below), then the rotation in two groups of four chunk pairs
// (c, c + 8), each with its eight table entries.
template <bool kCommon>
__device__ __forceinline__ void transform_half_row_d128(uint8_t* tile, int row, int h, int pos, const AttnParams& p) {
  constexpr int D = 128, NC = D / 8;
  float r = 1.0f;
  if (kCommon || p.use_norm) {
    uint64_t acc0 = 0, acc1 = 0;  // (P_{4h}, P_{4h+1}), (P_{4h+2}, P_{4h+3})
#pragma unroll
    for (int c = 0; c < NC; ++c) {
      const uint2 u = *reinterpret_cast<const uint2*>(tile + tile_off<D>(row, c) + 8 * h);
      const uint64_t a = bf16x2_to_f2<D>(u.x), b = bf16x2_to_f2<D>(u.y);
      acc0 = f2_fma(a, a, acc0);
      acc1 = f2_fma(b, b, acc1);
    }
    const uint64_t mine = f2_add(acc0, acc1);
    const uint64_t other = __shfl_xor_sync(0xffffffffu, mine, 1);
    const uint64_t e = h == 0 ? f2_add(mine, other) : f2_add(other, mine);
    const float ss = __fadd_rn(f2_lo(e), f2_hi(e));
    const float ms = __fmul_rn(ss, 1.0f / D);
    r = __frcp_rn(__fsqrt_rn(__fadd_rn(ms, p.eps)));  // = 1 / sqrt(.), both correctly rounded
  }
  if (p.rope != nullptr) {
    const uint64_t r2 = f2_pack(r, r), nr2 = f2_pack(-r, -r);
    const float4* src = p.rope + pos;
#pragma unroll
    for (int grp = 0; grp < 2; ++grp) {
      float4 cs[8];  // table entries k = 8 grp + kk, k = 2c + q
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const int k = 8 * grp + kk;
        const int i2 = 4 * (k >> 1) + 2 * h + (k & 1);
        cs[kk] = __ldg(src + static_cast<size_t>(i2) * p.rope_T);
      }
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) {
        const int c = 4 * grp + cc;
        const uint2 u1 = *reinterpret_cast<const uint2*>(tile + tile_off<D>(row, c) + 8 * h);
        const uint2 u2 = *reinterpret_cast<const uint2*>(tile + tile_off<D>(row, c + NC / 2) + 8 * h);
        const uint32_t w1[2] = {u1.x, u1.y}, w2[2] = {u2.x, u2.y};
        uint32_t wa[2], wb[2];
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          const float4 t = cs[2 * cc + q];
          const uint64_t cos2 = f2_pack(t.x, t.y), sin2 = f2_pack(t.z, t.w);
          const uint64_t c2 = f2_mul(cos2, r2), s2 = f2_mul(sin2, r2), sn2 = f2_mul(sin2, nr2);
          const uint64_t x1 = bf16x2_to_f2<D>(w1[q]), x2 = bf16x2_to_f2<D>(w2[q]);
          wa[q] = f2_to_bf16x2(f2_fma(x1, c2, f2_mul(x2, s2)));
          wb[q] = f2_to_bf16x2(f2_fma(x2, c2, f2_mul(x1, sn2)));
        }
        *reinterpret_cast<uint2*>(tile + tile_off<D>(row, c) + 8 * h) = make_uint2(wa[0], wa[1]);
        *reinterpret_cast<uint2*>(tile + tile_off<D>(row, c + NC / 2) + 8 * h) = make_uint2(wb[0], wb[1]);
      }
    }
  } else {
    const uint64_t r2 = f2_pack(r, r);
#pragma unroll
    for (int c = 0; c < NC; ++c) {
      uint2* w = reinterpret_cast<uint2*>(tile + tile_off<D>(row, c) + 8 * h);
      const uint2 u = *w;
      *w = make_uint2(f2_to_bf16x2(f2_mul(bf16x2_to_f2<D>(u.x), r2)), f2_to_bf16x2(f2_mul(bf16x2_to_f2<D>(u.y), r2)));
    }
  }
}

// kCommon: the call has the QK-norm on (the common case), so it is not tested at run time. (The RoPE
// test stays a run-time branch: with it compiled out the D = 64 kernel spills at the prologue's
// register share.)
template <int D, bool kCommon>
__device__ __forceinline__ void transform_half_row_inplace(uint8_t* tile, int row, int h, int pos, RopeHalf<D>& tab,
                                                           const AttnParams& p) {
  if constexpr (D == 128) {
    transform_half_row_d128<kCommon>(tile, row, h, pos, p);
    return;
  }
  constexpr int NC = D / 8;  // chunks per row; this thread owns 2 words (4 elements) of each
  uint64_t x[2 * NC];        // x[2c], x[2c+1]: elements 8c + 4h + {0,1} and {2,3} as fp32 pairs
#pragma unroll
  for (int c = 0; c < NC; ++c) {
    const uint2 u = *reinterpret_cast<const uint2*>(tile + tile_off<D>(row, c) + 8 * h);
    x[2 * c] = bf16x2_to_f2<D>(u.x);
    x[2 * c + 1] = bf16x2_to_f2<D>(u.y);
  }
  float r = 1.0f;
  if (kCommon || p.use_norm) {
    uint64_t acc0 = 0, acc1 = 0;  // (P_{4h}, P_{4h+1}), (P_{4h+2}, P_{4h+3})
#pragma unroll
    for (int c = 0; c < NC; ++c) {
      acc0 = f2_fma(x[2 * c], x[2 * c], acc0);
      acc1 = f2_fma(x[2 * c + 1], x[2 * c + 1], acc1);
    }
    const uint64_t mine = f2_add(acc0, acc1);  // h=0: (P0+P2, P1+P3); h=1: (P4+P6, P5+P7)
    const uint64_t other = __shfl_xor_sync(0xffffffffu, mine, 1);
    const uint64_t e = h == 0 ? f2_add(mine, other) : f2_add(other, mine);
    const float ss = __fadd_rn(f2_lo(e), f2_hi(e));
    const float ms = __fmul_rn(ss, 1.0f / D);
    r = __frcp_rn(__fsqrt_rn(__fadd_rn(ms, p.eps)));  // = 1 / sqrt(.), both correctly rounded
  }
  if (p.rope != nullptr) {
    // Loaded here rather than before the tile arrives: keeping both the fp32 row and the table
    // live across the wait does not fit the prologue's register share.
    tab.load(p, pos, h);
    const uint64_t r2 = f2_pack(r, r), nr2 = f2_pack(-r, -r);
    // pair i = 8c + 4h + 2q + e (c < NC/2, q, e in {0,1}) is element e of x[2c + q]; its partner
    // i + D/2 is element e of x[2(c + NC/2) + q]. Table entry k = 2c + q.
#pragma unroll
    for (int c = 0; c < NC / 2; ++c) {
      uint32_t wa[2], wb[2];
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const float4 t = tab.cs[2 * c + q];
        const uint64_t cos2 = f2_pack(t.x, t.y), sin2 = f2_pack(t.z, t.w);
        const uint64_t c2 = f2_mul(cos2, r2), s2 = f2_mul(sin2, r2), sn2 = f2_mul(sin2, nr2);
        const uint64_t x1 = x[2 * c + q], x2 = x[2 * (c + NC / 2) + q];
        wa[q] = f2_to_bf16x2(f2_fma(x1, c2, f2_mul(x2, s2)));
        wb[q] = f2_to_bf16x2(f2_fma(x2, c2, f2_mul(x1, sn2)));
      }
      *reinterpret_cast<uint2*>(tile + tile_off<D>(row, c) + 8 * h) = make_uint2(wa[0], wa[1]);
      *reinterpret_cast<uint2*>(tile + tile_off<D>(row, c + NC / 2) + 8 * h) = make_uint2(wb[0], wb[1]);
    }
  } else {
    const uint64_t r2 = f2_pack(r, r);
#pragma unroll
    for (int c = 0; c < NC; ++c)
      *reinterpret_cast<uint2*>(tile + tile_off<D>(row, c) + 8 * h) =
          make_uint2(f2_to_bf16x2(f2_mul(x[2 * c], r2)), f2_to_bf16x2(f2_mul(x[2 * c + 1], r2)));
  }
}

// The gate factor of the value-embedding gate for every (b, t, K/V head), one thread per (b, t):
// 2 * bf16(sigmoid(bf16(x[b, t, 0:32] . w[hk, 0:32]))). The habr "Autoresearch" listing computes it on
// bf16 tensors (CausalSelfAttention.forward, value residual), so the logit (a 32-term dot product
// accumulated in fp32) and the sigmoid (1 / (1 + exp(-logit)) with the accurate exp and a correctly
// rounded add and reciprocal) are each rounded to bf16; the factor 2 is exact.
__global__ void __launch_bounds__(256) ve_gate_kernel(AttnParams p) {
  const long long n = static_cast<long long>(p.B) * p.T;
  for (long long r = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; r < n;
       r += static_cast<long long>(gridDim.x) * blockDim.x) {
    const uint4* xr = reinterpret_cast<const uint4*>(p.xg + r * p.xg_stride);
    float xv[32];
#pragma unroll
    for (int c = 0; c < 4; ++c) bf16x8_to_f32(__ldg(xr + c), xv + 8 * c);
    for (int hk = 0; hk < p.Hkv; ++hk) {
      const uint4* wr = reinterpret_cast<const uint4*>(p.wg + static_cast<size_t>(hk) * 32);
      float acc = 0.f;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        float wv[8];
        bf16x8_to_f32(__ldg(wr + c), wv);
#pragma unroll
        for (int e = 0; e < 8; ++e) acc = fmaf(xv[8 * c + e], wv[e], acc);
      }
      const float lg = __bfloat162float(__float2bfloat16_rn(acc));
      const float sg = __bfloat162float(__float2bfloat16_rn(__frcp_rn(__fadd_rn(1.0f, expf(-lg)))));
      p.gate[r * p.Hkv + hk] = 2.0f * sg;
    }
  }
}


// Value-embedding gate of one V row in place, split over two threads like the prologue's K rows
// (thread h owns the 8 bytes at 8 h of every 16-byte chunk): v' = bf16(v + bf16(gate * ve)), with the
// row's gate factor from ve_gate_kernel (attn_common.cuh). gate * ve is exact in fp32 (a bf16 value
// times twice a bf16 value), so only its rounding and the sum's are steps of their own.
template <int D>
__device__ __forceinline__ void gate_half_row_inplace(uint8_t* tile, int row, int h, int pos, int b, int hk,
                                                      const AttnParams& p) {
  const size_t r = (static_cast<size_t>(b) * p.T + pos) * p.Hkv + hk;
  const float gate = __ldg(p.gate + r);
  const uint2* er = reinterpret_cast<const uint2*>(p.ve + r * D) + h;
  uint2 ev[D / 8];
#pragma unroll
  for (int c = 0; c < D / 8; ++c) ev[c] = __ldg(er + 2 * c);
#pragma unroll
  for (int c = 0; c < D / 8; ++c) {
    uint2* w = reinterpret_cast<uint2*>(tile + tile_off<D>(row, c) + 8 * h);
    const uint2 u = *w;
    const uint32_t in[2] = {u.x, u.y}, ew[2] = {ev[c].x, ev[c].y};
    uint32_t o[2];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const float v0 = __uint_as_float(in[k] << 16), v1 = __uint_as_float(in[k] & 0xFFFF0000u);
      const float e0 = __uint_as_float(ew[k] << 16), e1 = __uint_as_float(ew[k] & 0xFFFF0000u);
      const float p0 = __bfloat162float(__float2bfloat16_rn(gate * e0));
      const float p1 = __bfloat162float(__float2bfloat16_rn(gate * e1));
      o[k] = pack_bf16x2(__fadd_rn(v0, p0), __fadd_rn(v1, p1));
    }
    *w = make_uint2(o[0], o[1]);
  }
}

struct WsMaps {
  CUtensorMap q, k, v;  // 4-D (D, H, T, B) views, box (min(D, 64), 1, 128, 1), swizzled
  CUtensorMap out;      // the same view of the output, box (min(D, 64), 1, kOutRows, 1)
};

// Visible columns of one 32-column block as a bit mask (bit c set: column c visible), for the
// block-relative visible range [lo, hi].
__device__ __forceinline__ uint32_t block_vis(int lo, int hi) {
  const uint32_t upper = hi >= 31 ? 0xFFFFFFFFu : (hi < 0 ? 0u : (0xFFFFFFFFu >> (31 - hi)));
  const uint32_t lower = lo <= 0 ? 0xFFFFFFFFu : (lo > 31 ? 0u : (0xFFFFFFFFu << lo));
  return upper & lower;
}

// Columns whose bit is clear in `vis` -> -inf (no branches: one select per element).
__device__ __forceinline__ void mask_block(uint32_t (&s)[32], uint32_t vis) {
#pragma unroll
  for (int c = 0; c < 32; ++c) s[c] = (vis >> c) & 1u ? s[c] : 0xFF800000u;
}

// Max of one loaded 32-column block: the hardware-reduced value when no column is masked, else
// the max of the values after masking (which masks them in place).
__device__ __forceinline__ float block_max(uint32_t (&s)[32], float red, uint32_t vis) {
  if (vis == 0u) return -INFINITY;
  if (vis == 0xFFFFFFFFu) return red;
  mask_block(s, vis);
  float m0 = -INFINITY, m1 = -INFINITY, m2 = -INFINITY, m3 = -INFINITY;
#pragma unroll
  for (int c = 0; c < 32; c += 8) {
    m0 = fmax3(m0, __uint_as_float(s[c + 0]), __uint_as_float(s[c + 1]));
    m1 = fmax3(m1, __uint_as_float(s[c + 2]), __uint_as_float(s[c + 3]));
    m2 = fmax3(m2, __uint_as_float(s[c + 4]), __uint_as_float(s[c + 5]));
    m3 = fmax3(m3, __uint_as_float(s[c + 6]), __uint_as_float(s[c + 7]));
  }
  return fmax3(m0, m1, fmaxf(m2, m3));
}

// P = exp2(s * scale - m) of one block (masked columns hold -inf and give 0), packed to bf16 and
// stored into 16 TMEM columns at tP; returns the block's sum of P (fp32). A block with no visible
// column stores zeros. The exponentials stay scalar and are summed by a scalar tree: measured on one
// warp, that is faster than summing them as packed pairs, which costs register moves and a longer
// dependency chain.
__device__ __forceinline__ float exp_store(const uint32_t (&s)[32], bool empty, uint64_t scale2, uint64_t negm2,
                                           uint32_t tP) {
  uint32_t pk[16];
  float sum = 0.f;
  if (empty) {
#pragma unroll
    for (int c = 0; c < 16; ++c) pk[c] = 0u;
  } else {
    float p[32];
#pragma unroll
    for (int c = 0; c < 16; ++c) {
      const uint64_t x2 = f2_fma(f2_pack(__uint_as_float(s[2 * c]), __uint_as_float(s[2 * c + 1])), scale2, negm2);
      p[2 * c] = ex2_approx(f2_lo(x2));
      p[2 * c + 1] = ex2_approx(f2_hi(x2));
    }
    float t[16];
#pragma unroll
    for (int c = 0; c < 16; ++c) t[c] = p[2 * c] + p[2 * c + 1];
#pragma unroll
    for (int c = 0; c < 8; ++c) t[c] += t[c + 8];
#pragma unroll
    for (int c = 0; c < 4; ++c) t[c] += t[c + 4];
    sum = (t[0] + t[2]) + (t[1] + t[3]);
#pragma unroll
    for (int c = 0; c < 16; ++c) pk[c] = pack_bf16x2(p[2 * c], p[2 * c + 1]);
  }
  __syncwarp();  // the TMEM store is warp-collective; `empty` may differ between rows
  tmem_st16(tP, pk);
  return sum;
}

// Softmax of one S tile held in TMEM at tS for this thread's row (lane): the row sees columns
// lo..hi when `masked` (an unmasked tile: all 128). Writes P (bf16) over the upper half of the
// buffer, returns the row sum of P and sets the new reference max m_new and the factor alpha that
// rescales the previous O and l. `masked` is uniform over the warpgroup; the unmasked tiles skip
// the per-block mask tests at run time.
//
// Two passes over the four 32-column blocks of S: the row max, two blocks per TMEM round trip with
// the reducing load; then the exponentials one block per round trip, in the order 3, 2, 0, 1 so
// that S blocks 3 and 2 are read before P (16 columns per block, at column 64 + 16 b) covers them.
// The kernel is limited by instruction fetch more than by instruction count: this form keeps one
// copy of the exponential code and measured faster than handling two blocks per trip, which
// needs two copies; likewise one copy serves masked and unmasked tiles.
__device__ __forceinline__ float softmax_tile(bool masked, uint32_t tS, int lo, int hi, float scale, uint64_t scale2,
                                              float m_used, float& m_new, float& alpha) {
  float mx = -INFINITY;
#pragma unroll 1
  for (int hb = 0; hb < 4; hb += 2) {
    const uint32_t va = masked ? block_vis(lo - 32 * hb, hi - 32 * hb) : 0xFFFFFFFFu;
    const uint32_t vc = masked ? block_vis(lo - 32 * hb - 32, hi - 32 * hb - 32) : 0xFFFFFFFFu;
    uint32_t a[32], c[32];
    float ra = -INFINITY, rc = -INFINITY;
    __syncwarp();  // warp-collective TMEM loads after per-row branches
    tmem_ld32_max(tS + 32 * hb, a, ra);
    tmem_ld32_max(tS + 32 * hb + 32, c, rc);
    tmem_ld_wait();
    reg_fence<32>(a);
    reg_fence<32>(c);
    asm volatile("" : "+f"(ra), "+f"(rc));
    mx = fmax3(mx, block_max(a, ra, va), block_max(c, rc, vc));
  }
  const float m_tile = mx * scale;
  const bool grow = m_tile > m_used + kRescaleLog2 || (m_used == -INFINITY && m_tile > -INFINITY);
  m_new = grow ? m_tile : m_used;
  alpha = grow ? ex2_approx(m_used - m_new) : 1.0f;  // 0 when m_used = -inf
  const float m_use = m_new == -INFINITY ? 0.f : m_new;
  const uint64_t negm2 = f2_pack(-m_use, -m_use);
  float rowsum = 0.f;
#pragma unroll 1
  for (int i = 0; i < 4; ++i) {
    const int bk = i < 2 ? 3 - i : i - 2;
    const uint32_t v = masked ? block_vis(lo - 32 * bk, hi - 32 * bk) : 0xFFFFFFFFu;
    uint32_t a[32];
    __syncwarp();
    tmem_ld32(tS + 32 * bk, a);
    tmem_ld_wait();
    reg_fence<32>(a);
    if (v != 0xFFFFFFFFu) mask_block(a, v);
    rowsum += exp_store(a, v == 0u, scale2, negm2, tS + 64 + 16 * bk);
  }
  return rowsum;
}

// Softmax of one S tile against a fixed reference R (p.ref_log2 > 0): with the QK-norm on, every
// q^ and k^ row has norm at most sqrt(D), so |q^ . k^| <= D and every scaled score lies in [-R, R]
// for R just above sqrt(D) log2(e). P = exp2(s * scale - R) then lies in [2^-2R, 1]: no running
// maximum, no max pass and no O rescale are needed, and the result is the same softmax. The four
// 32-column blocks go in the order 3, 2, 0, 1 (P of block b is written at column 64 + 16 b, over S
// columns already read), and the TMEM load of the next block is issued before the exponentials of
// the current one so its latency overlaps them (two register buffers, one loop iteration per pair
// of blocks). Returns the row sum of P.
__device__ __forceinline__ float softmax_tile_fixed(bool masked, uint32_t tS, int lo, int hi, uint64_t scale2,
                                                    uint64_t negr2) {
  float rowsum = 0.f;
  uint32_t a[32], c[32];
  __syncwarp();
  tmem_ld32(tS + 96, a);  // block 3
#pragma unroll 1
  for (int k = 0; k < 2; ++k) {
    const int b0 = k == 0 ? 3 : 0, b1 = k == 0 ? 2 : 1;
    tmem_ld_wait();
    reg_fence<32>(a);
    __syncwarp();
    tmem_ld32(tS + 32 * b1, c);
    {
      const uint32_t v = masked ? block_vis(lo - 32 * b0, hi - 32 * b0) : 0xFFFFFFFFu;
      if (v != 0xFFFFFFFFu) mask_block(a, v);
      rowsum += exp_store(a, v == 0u, scale2, negr2, tS + 64 + 16 * b0);
    }
    tmem_ld_wait();
    reg_fence<32>(c);
    if (k == 0) {
      __syncwarp();
      tmem_ld32(tS, a);  // block 0, for the next iteration
    }
    {
      const uint32_t v = masked ? block_vis(lo - 32 * b1, hi - 32 * b1) : 0xFFFFFFFFu;
      if (v != 0xFFFFFFFFu) mask_block(c, v);
      rowsum += exp_store(c, v == 0u, scale2, negr2, tS + 64 + 16 * b1);
    }
  }
  return rowsum;
}

// kCommon: the call has the QK-norm on and no value-embedding gate (the common case); that
// instantiation carries no code for the other modes (the raw softmax with a running maximum and
// its O rescale, the prologue without the norm, the gate), which keeps the hot loops' code small.
template <int D, bool kCommon>
__global__ void __launch_bounds__(640, 1)
    attn_fwd_ws_kernel(const AttnParams p, const __grid_constant__ WsMaps maps, int* sched, int n_chunks) {
  using Cfg = WsCfg<D>;
  constexpr int TB = Cfg::kTileBytes;
  constexpr int S = Cfg::kStages;
  constexpr int NB = Cfg::kSBufs;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Cfg::kOffBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Cfg::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Cfg::kOffMisc + 4);
  volatile int* unit_id = reinterpret_cast<volatile int*>(smem + Cfg::kOffMisc + 8);  // [2]
  // [2] geometry of the unit in each slot, written by the producer with the unit id
  UnitGeom* unit_geo = reinterpret_cast<UnitGeom*>(smem + Cfg::kOffMisc + 16);
  auto bar = [&](int i) { return bars + i; };
  auto q_tile = [&](int slot, int t) { return smem + Cfg::kOffQ + (2 * slot + t) * TB; };
  auto k_tile = [&](int st) { return smem + Cfg::kOffK + st * TB; };
  auto v_tile = [&](int st) { return smem + Cfg::kOffV + st * TB; };
  // One 128-row tile by TMA: D > 64 goes as 64-column boxes into the 16 KB sub-tiles of the layout.
  constexpr int kBoxes = D > 64 ? D / 64 : 1;
  auto load_tile = [&](uint8_t* dst, const CUtensorMap* map, uint64_t* full, int h, int t, int b, uint64_t pol) {
#pragma unroll
    for (int x = 0; x < kBoxes; ++x) tma_load_4d_hint(dst + x * kTile * 128, map, full, 64 * x, h, t, b, pol);
  };

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int n_qb = (p.T + 2 * kTile - 1) / (2 * kTile);

  if (tid == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(Cfg::kBarQFull + i), 1);
      mbar_init(bar(Cfg::kBarQReady + i), 8);
      mbar_init(bar(Cfg::kBarQEmpty + i), kQEmptyArrivals);
      mbar_init(bar(Cfg::kBarUnit + i), 1);
    }
    for (int i = 0; i < 4; ++i) {
      mbar_init(bar(Cfg::kBarSFull + i), 1);
      mbar_init(bar(Cfg::kBarPFull + i), 4);
      mbar_init(bar(Cfg::kBarPVDone + i), 1);
    }
    for (int i = 0; i < S; ++i) {
      mbar_init(bar(Cfg::kBarKFull + i), 1);
      mbar_init(bar(Cfg::kBarKReady + i), 8);
      mbar_init(bar(Cfg::kBarVFull + i), 1);
      mbar_init(bar(Cfg::kBarKFree + i), 1);
      mbar_init(bar(Cfg::kBarVFree + i), 2);
    }
    for (int i = 0; i < NB; ++i) mbar_init(bar(Cfg::kBarBufFree + i), 1);
    for (int i = 0; i < 3; ++i) mbar_init(bar(Cfg::kBarFinal + i), 1);
    for (int i = 0; i < S; ++i) mbar_init(bar(Cfg::kBarVReady + i), 8);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 17) {
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

  if (warp >= 16) {
    regs_dec<64>();
  }
  if (warp == 16) {
    if (lane == 0) {
      // ---------------- producer: tickets and TMA loads ----------------
      prefetch_tmap(&maps.q);
      prefetch_tmap(&maps.k);
      prefetch_tmap(&maps.v);
      const uint64_t pol_stream = policy_evict_first();
      const uint64_t pol_keep = policy_evict_last();
      int q_armed[2] = {-1, -1};  // parity of the last armed phase of each Q barrier (for draining)
      uint32_t kcnt = 0;          // K/V stage loads issued
      bool ok = true;
      // A ticket is a chunk of consecutive query blocks of one head, taken top down: all of them for
      // heads 0 .. n_long - 1, then blocks qb and qb - 1 of the other heads, heaviest pairs of every
      // head first. The units of a chunk run back to back on this CTA, and each shares the key tiles
      // that it and the next one need through the ring (shared_steps).
      const int n_bh = p.B * p.H;
      int c_bh = 0, c_qb = -1, c_left = 0;  // the current chunk: head, next query block, units left
      bool c_first = false;                 // the next unit is the first of its chunk
      UnitGeom g;
      g.r_out = 0;
      for (uint32_t ul = 0;; ++ul) {
        const int slot = ul % Cfg::kQSlots;
        const uint32_t uph = (ul / Cfg::kQSlots) & 1;
        if (!mbar_wait_or_abort(bar(Cfg::kBarQEmpty + slot), uph ^ 1, abort_flag)) {
          ok = false;
          break;
        }
        int unit = -1;
        if (c_left == 0) {
          const int c = atomicAdd(sched, 1);
          if (c < p.n_long) {
            // a whole head, every query block top down
            c_bh = c;
            c_qb = n_qb - 1;
            c_left = n_qb;
          } else if (c < n_chunks) {
            // pairs of the other heads: groups of head_group heads in turn; inside a group the
            // heaviest pair of every head first, then the next pair of every head, ...
            const int cp = c - p.n_long;
            const int cpb = (n_qb + 1) / 2;  // pairs per head
            const int grp = cp / (p.head_group * cpb);
            const int rem = cp - grp * p.head_group * cpb;
            const int gsize = min(p.head_group, n_bh - p.n_long - grp * p.head_group);
            const int rank = rem / gsize;
            c_bh = p.n_long + grp * p.head_group + (rem - rank * gsize);
            c_qb = n_qb - 1 - 2 * rank;
            c_left = c_qb >= 1 ? 2 : 1;
          }
          c_first = true;
        }
        if (c_left > 0) {
          const int r_in = g.r_out;  // the previous unit (same chunk) left that many steps
          unit_geom(p, c_bh, c_qb, g);
          unit = c_bh * n_qb + c_qb;
          g.r_in = c_first ? 0 : r_in;
          c_first = false;
          if (c_left >= 2) {
            UnitGeom nb;
            unit_geom(p, c_bh, c_qb - 1, nb);
            g.r_out = shared_steps<S>(g, nb);
          }
          --c_left;
          --c_qb;
          unit_geo[slot] = g;  // read by the other roles after the unit barrier
        }
        unit_id[slot] = unit;
        mbar_arrive(bar(Cfg::kBarUnit + slot));
        if (unit < 0) {
          mbar_arrive(bar(Cfg::kBarQFull + slot));
          break;
        }
        const bool two = g.valid(1);
        mbar_arrive_expect_tx(bar(Cfg::kBarQFull + slot), (two ? 2 : 1) * TB);
        q_armed[slot] = static_cast<int>(uph);
        load_tile(q_tile(slot, 0), &maps.q, bar(Cfg::kBarQFull + slot), g.h, g.qs0, g.b, pol_stream);
        if (two)
          load_tile(q_tile(slot, 1), &maps.q, bar(Cfg::kBarQFull + slot), g.h, g.qs0 + kTile, g.b, pol_stream);
        // key steps from ke_all down; the first r_in are already resident (no load)
        for (int i = g.r_in; i < g.n_steps(); ++i, ++kcnt) {
          const int j = g.ke_all - i;
          const int st = kcnt % S;
          const uint32_t ph = (kcnt / S) & 1;
          if (!mbar_wait_or_abort(bar(Cfg::kBarKFree + st), ph ^ 1, abort_flag) ||
              !mbar_wait_or_abort(bar(Cfg::kBarVFree + st), ph ^ 1, abort_flag)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(bar(Cfg::kBarKFull + st), TB);
          load_tile(k_tile(st), &maps.k, bar(Cfg::kBarKFull + st), g.hk, j * kTile, g.b, pol_keep);
          mbar_arrive_expect_tx(bar(Cfg::kBarVFull + st), TB);
          load_tile(v_tile(st), &maps.v, bar(Cfg::kBarVFull + st), g.hk, j * kTile, g.b, pol_keep);
        }
        if (!ok) break;
      }
      if (!ok) {
        fail();
        // Drain: every TMA load this thread issued must land before the CTA exits. Only the last
        // S K/V loads can still be in flight (each earlier one was consumed before its stage was
        // reloaded); load n went to stage n % S, phase n / S.
        const uint32_t first = kcnt > static_cast<uint32_t>(S) ? kcnt - S : 0u;
#pragma unroll 1
        for (uint32_t m = 2 * first; m < 2 * kcnt + 2; ++m) {
          int b, par;
          if (m >= 2 * kcnt) {
            b = Cfg::kBarQFull + static_cast<int>(m - 2 * kcnt);
            par = q_armed[m - 2 * kcnt];
          } else {
            const uint32_t n = m >> 1;
            b = ((m & 1) ? Cfg::kBarVFull : Cfg::kBarKFull) + static_cast<int>(n % S);
            par = static_cast<int>((n / S) & 1);
          }
          if (par >= 0) mbar_wait(bar(b), static_cast<uint32_t>(par));
        }
      }
      // The last CTA to leave resets the ticket counters for the next launch on this slot.
      __threadfence();
      const int done = atomicAdd(sched + 1, 1);
      if (done == static_cast<int>(gridDim.x) - 1) {
        atomicExch(sched, 0);
        atomicExch(sched + 1, 0);
      }
    }
  } else if (warp == 17) {
    if (lane == 0) {
      // ---------------- S issuer: S = Q^ K^^T jobs in stream order ----------------
      using G = TileGeom<D>;
      constexpr uint32_t idesc_s = make_idesc_bf16(128, 128, false);
      bool ok = true;
      uint32_t gS = 0, kc = 0, scnt0 = 0, scnt1 = 0;
      for (uint32_t ul = 0; ok; ++ul) {
        const int slot = ul % Cfg::kQSlots;
        const uint32_t uph = (ul / Cfg::kQSlots) & 1;
        if (!mbar_wait_or_abort(bar(Cfg::kBarUnit + slot), uph, abort_flag)) { ok = false; break; }
        const int unit = unit_id[slot];
        if (unit < 0) break;
        if (!mbar_wait_or_abort(bar(Cfg::kBarQReady + slot), uph, abort_flag)) { ok = false; break; }
        const UnitGeom g = unit_geo[slot];
        const int n_st = g.n_steps();
        for (int i = 0; i < n_st && ok; ++i) {
          const int j = g.ke_all - i;
          // ring position of step i: a resident step sits where the previous unit loaded it (its
          // K^-ready phase is complete and the stage is not reloaded before this unit frees it)
          const uint32_t pos = i < g.r_in ? kc - g.r_in + i : kc++;
          const int st = pos % S;
          if (!mbar_wait_or_abort(bar(Cfg::kBarKReady + st), (pos / S) & 1, abort_flag)) { ok = false; break; }
          const uint32_t ka = smem_u32(k_tile(st));
#pragma unroll 1
          for (int t = 0; t < 2; ++t) {
            if (!g.has(t, j)) continue;
            const int b = gS % NB;
            uint32_t& sc = t == 0 ? scnt0 : scnt1;
            // S job n of tile t (on S-done slot n & 1) waits for the buffer's previous P.V and for the
            // tile's P.V job n - 2. That P.V needed P of job n - 2, so the tile's softmax has consumed
            // the S-done slot of job n - 2; and a softmax that waits for P.V job n - 1 (O rescale,
            // epilogue) knows that job n - 3 has completed and job n + 1 cannot have: every two-slot
            // parity wait is exact.
            if (!mbar_wait_or_abort(bar(Cfg::kBarBufFree + b), ((gS / NB) & 1) ^ 1, abort_flag) ||
                (sc >= 2 && !mbar_wait_or_abort(bar(Cfg::kBarPVDone + 2 * t + (sc & 1)), ((sc - 2) >> 1) & 1,
                                                abort_flag))) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t qa = smem_u32(q_tile(slot, t));
#pragma unroll
            for (int ks = 0; ks < G::kKSteps; ++ks) {
              const uint64_t ad = make_sdesc(qa + G::kstep_off(ks), 16, G::kSBO, G::kSwizzle);
              const uint64_t bd = make_sdesc(ka + G::kstep_off(ks), 16, G::kSBO, G::kSwizzle);
              umma_ss(tmem + Cfg::col_buf(b), ad, bd, idesc_s, ks > 0 ? 1u : 0u);
            }
            umma_commit(bar(Cfg::kBarSFull + 2 * t + (sc & 1)));
            ++sc;
            ++gS;
          }
          // K^ of this stage no longer read (unless the next unit reuses it)
          if (ok && i < n_st - g.r_out) umma_commit(bar(Cfg::kBarKFree + st));
        }
        // the unit's Q^ tiles are no longer read once its last S job completes
        if (ok) umma_commit(bar(Cfg::kBarQEmpty + slot));
      }
      if (!ok) fail();
      umma_commit(bar(Cfg::kBarFinal + 0));
      mbar_wait(bar(Cfg::kBarFinal + 0), 0);
    }
  } else if (warp == 18 || warp == 19) {
    if (lane == 0) {
      // ---------------- P.V issuer of query tile t: O_t += P V, in order ----------------
      using G = TileGeom<D>;
      constexpr uint32_t idesc_o = make_idesc_bf16(128, D, true);
      const int t = warp - 18;
      bool ok = true;
      uint32_t gS = 0, kc = 0, pcnt = 0;
      for (uint32_t ul = 0; ok; ++ul) {
        const int slot = ul % Cfg::kQSlots;
        const uint32_t uph = (ul / Cfg::kQSlots) & 1;
        if (!mbar_wait_or_abort(bar(Cfg::kBarUnit + slot), uph, abort_flag)) { ok = false; break; }
        const int unit = unit_id[slot];
        if (unit < 0) break;
        const UnitGeom g = unit_geo[slot];
        // The slot's unit id and geometry have been read (one of the arrivals that free the slot).
        mbar_arrive(bar(Cfg::kBarQEmpty + slot));
        const int n_st = g.n_steps();
        for (int i = 0; i < n_st; ++i) {
          const int j = g.ke_all - i;
          const bool h0 = g.has(0, j), h1 = g.has(1, j);
          const uint32_t gj = gS + (t == 1 && h0 ? 1u : 0u);
          gS += (h0 ? 1u : 0u) + (h1 ? 1u : 0u);
          const uint32_t pos = i < g.r_in ? kc - g.r_in + i : kc++;  // ring position (see the S issuer)
          const int st = pos % S;
          const bool release = i < n_st - g.r_out;  // not kept for the next unit
          // Every load's V phase is observed (and released, at its last use) by both issuers, active
          // or not, so the stage's barriers never run two phases ahead of either of them.
          // a gated call's V tile is read once the prologue has applied the gate to it
          if (!mbar_wait_or_abort(bar((!kCommon && p.ve != nullptr ? Cfg::kBarVReady : Cfg::kBarVFull) + st), (pos / S) & 1,
                                  abort_flag)) {
            ok = false;
            break;
          }
          if (!(t == 0 ? h0 : h1)) {
            if (release) mbar_arrive(bar(Cfg::kBarVFree + st));
            continue;
          }
          const int b = gj % NB;
          // P of this tile's job k, on slot k & 1: P of job k + 2 needs S job k + 2, which waits for
          // this P.V, so the slot is never two phases ahead of this wait.
          const uint32_t k = pcnt++;
          if (!mbar_wait_or_abort(bar(Cfg::kBarPFull + 2 * t + (k & 1)), (k >> 1) & 1, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t va = smem_u32(v_tile(st));
          const uint32_t pa = tmem + Cfg::col_buf(b) + 64;
          const bool first = j == g.ke(t);  // the unit's first P.V of this tile starts O_t
#pragma unroll
          for (int ks = 0; ks < 8; ++ks) {
            // V as the MN-major B operand; for D = 128 its two 64-column sub-tiles are kBytes / 2 apart
            const uint64_t bd = make_sdesc(va + ks * 16 * G::kRowBytes, D >= 128 ? G::kBytes / 2 : 16, G::kSBO,
                                           G::kSwizzle);
            umma_ts(tmem + Cfg::col_o(t), pa + ks * 8, bd, idesc_o, (!first || ks > 0) ? 1u : 0u);
          }
          umma_commit(bar(Cfg::kBarBufFree + b));
          umma_commit(bar(Cfg::kBarPVDone + 2 * t + (k & 1)));
          if (release) umma_commit(bar(Cfg::kBarVFree + st));
        }
      }
      if (!ok) fail();
      umma_commit(bar(Cfg::kBarFinal + 1 + t));
      mbar_wait(bar(Cfg::kBarFinal + 1 + t), 0);
    }
  } else if (warp >= 8) {
    regs_dec<80>();
    // ---------------- prologue: QK-norm + RoPE in place, two threads per row ----------------
    const int pr = tid - 256;       // 0..255
    const int r = pr >> 1;          // row of the tile
    const int h = pr & 1;           // half of the row
    uint32_t kcnt = 0;
    bool ok = true;
    RopeHalf<D> tab;
    for (uint32_t ul = 0; ok; ++ul) {
      const int slot = ul % Cfg::kQSlots;
      const uint32_t uph = (ul / Cfg::kQSlots) & 1;
      ok = __all_sync(0xffffffffu, mbar_wait_or_abort(bar(Cfg::kBarQFull + slot), uph, abort_flag));
      if (!ok) break;
      const int unit = unit_id[slot];
      if (unit < 0) break;
      const UnitGeom g = unit_geo[slot];
      // jobs 0, 1: the two Q tiles; then the K tiles the producer loads (not the resident ones),
      // from key step r_in on: step i holds key tile ke_all - i
      const int n_jobs = 2 + g.n_steps() - g.r_in;
#pragma unroll 1
      for (int jb = 0; jb < n_jobs; ++jb) {
        const bool is_q = jb < 2;
        if (is_q && !g.valid(jb)) {
          if (jb == 1 && lane == 0) mbar_arrive(bar(Cfg::kBarQReady + slot));
          continue;
        }
        const int st = kcnt % S;
        const int pos = is_q ? g.qs0 + kTile * jb + r : (g.ke_all - (g.r_in + jb - 2)) * kTile + r;
        uint8_t* tile = is_q ? q_tile(slot, jb) : k_tile(st);
        if (!is_q) {
          ok = __all_sync(0xffffffffu, mbar_wait_or_abort(bar(Cfg::kBarKFull + st), (kcnt / S) & 1, abort_flag));
          if (!ok) break;
        }
        transform_half_row_inplace<D, kCommon>(tile, r, h, pos < p.T ? pos : 0, tab, p);
        fence_proxy_async_smem();
        __syncwarp();
        if (is_q) {
          if (jb == 1 && lane == 0) mbar_arrive(bar(Cfg::kBarQReady + slot));
        } else {
          if (lane == 0) mbar_arrive(bar(Cfg::kBarKReady + st));
          if (!kCommon && p.ve != nullptr) {
            // the value-embedding gate on the same step's V tile, in place
            ok = __all_sync(0xffffffffu, mbar_wait_or_abort(bar(Cfg::kBarVFull + st), (kcnt / S) & 1, abort_flag));
            if (!ok) break;
            if (pos < p.T) gate_half_row_inplace<D>(v_tile(st), r, h, pos, g.b, g.hk, p);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(Cfg::kBarVReady + st));
          }
          ++kcnt;
        }
      }
    }
    if (!ok && lane == 0) fail();
  } else {
    regs_inc<128>();
    // ---------------- softmax + epilogue of query tile t ----------------
    const int t = warp >> 2;
    const int r = tid & 127;                                  // row in the tile = TMEM lane
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tO = tmem + lane_base + Cfg::col_o(t);
    const float scale = p.scale_log2;
    const uint64_t scale2 = f2_pack(scale, scale);
    const bool fixed_ref = kCommon || p.ref_log2 > 0.f;
    const uint64_t negr2 = f2_pack(-p.ref_log2, -p.ref_log2);
    uint32_t n = 0;   // P tiles written so far by this warpgroup (all units)
    uint32_t gS = 0;  // global S-job index, counted over both query tiles (as the MMA issuer does)
    bool ok = true;
    for (uint32_t ul = 0; ok; ++ul) {
      const int slot = ul % Cfg::kQSlots;
      const uint32_t uph = (ul / Cfg::kQSlots) & 1;
      ok = __all_sync(0xffffffffu, mbar_wait_or_abort(bar(Cfg::kBarUnit + slot), uph, abort_flag));
      if (!ok) break;
      const int unit = unit_id[slot];
      if (unit < 0) break;
      const UnitGeom g = unit_geo[slot];
      // the slot's unit id and geometry have been read (the arrival releases the reads)
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(Cfg::kBarQEmpty + slot));
      const int qs = g.qs0 + kTile * t;
      const int i_row = qs + r;
      float m_used = fixed_ref ? p.ref_log2 : -INFINITY;  // reference max of this row (log2 units)
      float l_run = 0.f;         // sum of exp2(score - m_used)
      for (int j = g.ke_all; j >= g.kb_all; --j) {  // key steps downwards, as the MMA issuers
        const bool h0 = g.has(0, j), h1 = g.has(1, j);
        const uint32_t gj = gS + (t == 1 && h0 ? 1u : 0u);
        gS += (h0 ? 1u : 0u) + (h1 ? 1u : 0u);
        if (!(t == 0 ? h0 : h1)) continue;
        const int k0 = j * kTile;
        const int b = gj % NB;
        const uint32_t tS = tmem + lane_base + Cfg::col_buf(b);
        // visible columns of this row in this tile: lo <= c <= hi
        int lo = 0, hi = kTile - 1;
        const bool masked = tile_needs_mask(p, qs, k0);  // same for the whole warpgroup
        if (masked) {
          lo = p.window >= 0 ? i_row - p.window - k0 : -1;
          hi = p.causal ? i_row - k0 : (p.window >= 0 ? i_row + p.window - k0 : kTile);
          hi = min(hi, p.T - 1 - k0);
        }
        // S of this tile's n-th job, on slot n & 1: S job n + 2 is issued only after this job's P.V,
        // which needs this job's P, so the slot is never two phases ahead of this wait.
        ok = __all_sync(0xffffffffu,
                        mbar_wait_or_abort(bar(Cfg::kBarSFull + 2 * t + (n & 1)), (n >> 1) & 1, abort_flag));
        if (!ok) break;
        tc_fence_after();

        float m_new = m_used, alpha = 1.0f;
        const float rowsum = fixed_ref ? softmax_tile_fixed(masked, tS, lo, hi, scale2, negr2)
                                       : softmax_tile(masked, tS, lo, hi, scale, scale2, m_used, m_new, alpha);
        // O rescale (running maximum only, rare): after the tile's previous P.V job (n - 1) has
        // completed; the next one is issued only after this job's P is announced.
        if (!fixed_ref && j < g.ke(t) && __any_sync(0xffffffffu, alpha != 1.0f)) {  // not the unit's first job
          ok = __all_sync(0xffffffffu, mbar_wait_or_abort(bar(Cfg::kBarPVDone + 2 * t + ((n - 1) & 1)),
                                                          ((n - 1) >> 1) & 1, abort_flag));
          if (!ok) break;
          tc_fence_after();
          uint32_t o[32];
#pragma unroll 1
          for (int cc = 0; cc < D / 32; ++cc) {
            tmem_ld32(tO + 32 * cc, o);
            tmem_ld_wait();
            reg_fence<32>(o);
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            tmem_st32(tO + 32 * cc, o);
          }
        }
        l_run = l_run * alpha + rowsum;
        m_used = m_new;
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(Cfg::kBarPFull + 2 * t + (n & 1)));
        ++n;
      }
      if (!ok) break;
      if (!g.valid(t)) continue;  // this query tile lies past T
      // ---- epilogue: O / l -> bf16; each warp stages its 32 rows and stores them by TMA; LSE ----
      ok = __all_sync(0xffffffffu, mbar_wait_or_abort(bar(Cfg::kBarPVDone + 2 * t + ((n - 1) & 1)),
                                                      ((n - 1) >> 1) & 1, abort_flag));
      if (!ok) break;
      tc_fence_after();
      const float inv_l = l_run > 0.f ? __frcp_rn(l_run) : 0.f;  // = 1 / l_run, correctly rounded
      const bool row_in = i_row < p.T;
      const int row0 = qs + kOutRows * (warp & 3);  // first row of this warp's box
      uint8_t* stg = smem + Cfg::kOffOut + warp * Cfg::kOutBytes;
      constexpr int kBoxCols = D > 64 ? 64 : D;
#pragma unroll 1
      for (int x = 0; x < kBoxes; ++x) {
        // the buffer is free once this warp's previous store from it has been read
        if (lane == 0) bulk_wait_group_read0();
        __syncwarp();
#pragma unroll 1
        for (int cc = 0; cc < kBoxCols / 32; ++cc) {
          uint32_t o[32];
          tmem_ld32(tO + kBoxCols * x + 32 * cc, o);
          tmem_ld_wait();
          reg_fence<32>(o);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint4 u;
            u.x = pack_bf16x2(__uint_as_float(o[q * 8 + 0]) * inv_l, __uint_as_float(o[q * 8 + 1]) * inv_l);
            u.y = pack_bf16x2(__uint_as_float(o[q * 8 + 2]) * inv_l, __uint_as_float(o[q * 8 + 3]) * inv_l);
            u.z = pack_bf16x2(__uint_as_float(o[q * 8 + 4]) * inv_l, __uint_as_float(o[q * 8 + 5]) * inv_l);
            u.w = pack_bf16x2(__uint_as_float(o[q * 8 + 6]) * inv_l, __uint_as_float(o[q * 8 + 7]) * inv_l);
            *reinterpret_cast<uint4*>(stg + out_stage_off<D>(lane, 4 * cc + q)) = u;
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0 && row0 < p.T) {
          tma_store_4d(&maps.out, stg, kBoxCols * x, g.h, row0, g.b);
          bulk_commit_group();
        }
      }
      if (p.lse != nullptr && row_in) {
        const float m_fin = m_used == -INFINITY ? 0.f : m_used;
        p.lse[(static_cast<size_t>(g.b) * p.H + g.h) * p.T + i_row] = (m_fin + __log2f(l_run)) * 0.69314718055994531f;
      }
    }
    if (!ok && lane == 0) fail();
    if (lane == 0) bulk_wait_group0();  // this warp's output stores are complete
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 17) {
    tc_fence_after();
    tmem_dealloc(tmem, Cfg::kTmemCols);
  }
}

}  // namespace swa
