// Attention forward, synchronous single-warpgroup version.
//
// One CTA of 128 threads per (b, h, 128-row query tile); thread t owns query row t of the tile
// and TMEM lane t. Per key tile: every thread normalises and rotates one K row and copies one V
// row into swizzled shared memory, thread 0 issues S = Q^ K^^T (tcgen05, accumulator in TMEM),
// every thread runs the online softmax on its row of S and writes P (bf16) back into TMEM, and
// thread 0 issues O += P V with P read from TMEM. Nothing overlaps; this kernel is the
// plain-structure twin of the pipelined kernel, kept as a second, independently structured GPU
// path for cross-checks.
#pragma once
#include "attn_common.cuh"

namespace swa {

template <int D>
struct SimpleCfg {
  using G = TileGeom<D>;
  static constexpr int kThreads = 128;
  static constexpr uint32_t kColS = 0;    // S: 128 fp32 columns
  static constexpr uint32_t kColP = 128;  // P: 128 bf16 = 64 columns
  static constexpr uint32_t kColO = 192;  // O: D fp32 columns
  static constexpr uint32_t kTmemCols = (kColO + D) <= 256 ? 256 : 512;
  static constexpr int kSmemTiles = 3 * G::kBytes;
  // Requested dynamic shared memory also bounds residency so that resident CTAs never ask for
  // more than the 512 TMEM columns of an SM (2 CTAs of 256 columns, or 1 of 512).
  static constexpr int kSmemFloor = kTmemCols == 256 ? 80 * 1024 : 120 * 1024;
  static constexpr int kSmemBytes = (kSmemTiles + 1024 + 64) > kSmemFloor ? (kSmemTiles + 1024 + 64) : kSmemFloor;
};

template <int D>
__global__ void __launch_bounds__(128, 1) attn_fwd_simple_kernel(const AttnParams p) {
  using Cfg = SimpleCfg<D>;
  using G = TileGeom<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  uint8_t* sQ = smem;
  uint8_t* sK = smem + G::kBytes;
  uint8_t* sV = smem + 2 * G::kBytes;
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + 3 * G::kBytes);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + 1);
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int qt = blockIdx.x % p.n_qtiles;
  const int bh = blockIdx.x / p.n_qtiles;
  const int h = bh % p.H;
  const int b = bh / p.H;
  const int T = p.T;
  const int q0 = qt * kTile;
  const size_t row_stride = static_cast<size_t>(p.H) * D;  // elements between consecutive t
  const size_t head_base = static_cast<size_t>(b) * T * row_stride + static_cast<size_t>(h) * D;
  // K/V rows: Hkv heads per position; this query head reads K/V head h / kv_group
  const size_t kv_stride = static_cast<size_t>(p.Hkv) * D;
  const size_t kv_base = static_cast<size_t>(b) * T * kv_stride + static_cast<size_t>(h / p.kv_group) * D;

  if (tid == 0) {
    mbar_init(bar, 1);
    *abort_flag = 0;
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

  // ---- Q tile: load, normalise, rotate, store swizzled ----
  {
    const int i = q0 + tid;
    uint32_t w[D / 2];
    const uint4* src = reinterpret_cast<const uint4*>(p.q + head_base + static_cast<size_t>(i) * row_stride);
#pragma unroll
    for (int ch = 0; ch < D / 8; ++ch) set_chunk<D>(w, ch, i < T ? __ldg(src + ch) : make_uint4(0, 0, 0, 0));
    qk_row_transform_packed<D>(w, i < T ? i : 0, p.rope, p.rope_T, p.use_norm, p.eps);
#pragma unroll
    for (int ch = 0; ch < D / 8; ++ch) *reinterpret_cast<uint4*>(sQ + tile_off<D>(tid, ch)) = get_chunk<D>(w, ch);
  }

  // ---- key-tile range of this query tile ----
  const int q_last = min(T - 1, q0 + kTile - 1);
  const int k_lo = p.window >= 0 ? max(0, q0 - p.window) : 0;
  const int k_hi = p.causal ? q_last : (p.window >= 0 ? min(T - 1, q_last + p.window) : T - 1);
  const int kt_begin = k_lo / kTile, kt_end = k_hi / kTile;  // inclusive

  constexpr uint32_t idesc_s = make_idesc_bf16(128, 128, false);
  constexpr uint32_t idesc_o = make_idesc_bf16(128, D, true);
  const uint32_t sQa = smem_u32(sQ), sKa = smem_u32(sK), sVa = smem_u32(sV);

  float m_run = -INFINITY;  // running max of scaled scores (log2 units)
  float l_run = 0.f;        // running sum of exp2(score - m_run)
  uint32_t phase = 0;
  const int i_row = q0 + tid;
  bool ok = true;

  for (int kt = kt_begin; kt <= kt_end; ++kt) {
    const int k0 = kt * kTile;
    // ---- K row (normalise + rotate) and V row into shared memory ----
    {
      const int j = k0 + tid;
      uint32_t w[D / 2];
      const uint4* src = reinterpret_cast<const uint4*>(p.k + kv_base + static_cast<size_t>(j) * kv_stride);
#pragma unroll
      for (int ch = 0; ch < D / 8; ++ch) set_chunk<D>(w, ch, j < T ? __ldg(src + ch) : make_uint4(0, 0, 0, 0));
      qk_row_transform_packed<D>(w, j < T ? j : 0, p.rope, p.rope_T, p.use_norm, p.eps);
#pragma unroll
      for (int ch = 0; ch < D / 8; ++ch) *reinterpret_cast<uint4*>(sK + tile_off<D>(tid, ch)) = get_chunk<D>(w, ch);
      const uint4* vsrc = reinterpret_cast<const uint4*>(p.v + kv_base + static_cast<size_t>(j) * kv_stride);
#pragma unroll
      for (int ch = 0; ch < D / 8; ++ch) {
        const uint4 u = j < T ? __ldg(vsrc + ch) : make_uint4(0, 0, 0, 0);
        *reinterpret_cast<uint4*>(sV + tile_off<D>(tid, ch)) = u;
      }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();

    // ---- S = Q^ K^^T ----
    if (tid == 0) {
      tc_fence_after();
#pragma unroll
      for (int ks = 0; ks < G::kKSteps; ++ks) {
        const uint64_t ad = make_sdesc(sQa + G::kstep_off(ks), 16, G::kSBO, G::kSwizzle);
        const uint64_t bd = make_sdesc(sKa + G::kstep_off(ks), 16, G::kSBO, G::kSwizzle);
        umma_ss(tmem + Cfg::kColS, ad, bd, idesc_s, ks > 0 ? 1u : 0u);
      }
      umma_commit(bar);
    }
    if (!mbar_wait(bar, phase)) {
      report_error(p.err, kDevErrTimeout);
      *abort_flag = 1;
    }
    phase ^= 1;
    tc_fence_after();

    // ---- online softmax on this thread's row ----
    uint32_t s[128];
#pragma unroll
    for (int c = 0; c < 4; ++c) tmem_ld32(tmem + lane_base + Cfg::kColS + 32 * c, s + 32 * c);
    tmem_ld_wait();
    reg_fence<128>(s);

    float mx = -INFINITY;
#pragma unroll
    for (int c = 0; c < 128; ++c) {
      float sc = __uint_as_float(s[c]) * p.scale_log2;
      if (!key_visible(i_row, k0 + c, T, p.window, p.causal)) sc = -INFINITY;
      s[c] = __float_as_uint(sc);
      mx = fmaxf(mx, sc);
    }
    const float m_new = fmaxf(m_run, mx);
    const float m_use = m_new == -INFINITY ? 0.f : m_new;
    const float alpha = ex2_approx(m_run - m_use);  // 0 when m_run = -inf
    float rowsum = 0.f;
    uint32_t pk[64];
#pragma unroll
    for (int c = 0; c < 64; ++c) {
      const float p0 = ex2_approx(__uint_as_float(s[2 * c]) - m_use);
      const float p1 = ex2_approx(__uint_as_float(s[2 * c + 1]) - m_use);
      rowsum += p0 + p1;
      pk[c] = pack_bf16x2(p0, p1);
    }
    l_run = l_run * alpha + rowsum;
    m_run = m_new;
    tmem_st32(tmem + lane_base + Cfg::kColP, pk);
    tmem_st32(tmem + lane_base + Cfg::kColP + 32, pk + 32);
    // tcgen05.ld/st are warp-collective: the rescale runs for the whole warp when any row of
    // it needs it (rows with alpha == 1 multiply by 1).
    if (kt > kt_begin && __any_sync(0xffffffffu, alpha != 1.0f)) {
      uint32_t o[D];
#pragma unroll
      for (int c = 0; c < D / 32; ++c) tmem_ld32(tmem + lane_base + Cfg::kColO + 32 * c, o + 32 * c);
      tmem_ld_wait();
      reg_fence<D>(o);
#pragma unroll
      for (int c = 0; c < D; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * alpha);
#pragma unroll
      for (int c = 0; c < D / 32; ++c) tmem_st32(tmem + lane_base + Cfg::kColO + 32 * c, o + 32 * c);
    }
    tmem_st_wait();
    tc_fence_before();
    __syncthreads();
    if (*abort_flag) {
      ok = false;
      break;
    }

    // ---- O += P V ----
    if (tid == 0) {
      tc_fence_after();
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        const uint64_t bd = make_sdesc(sVa + ks * 16 * G::kRowBytes, D >= 128 ? G::kBytes / 2 : 16, G::kSBO,
                                       G::kSwizzle);
        umma_ts(tmem + Cfg::kColO, tmem + Cfg::kColP + ks * 8, bd, idesc_o, (kt > kt_begin || ks > 0) ? 1u : 0u);
      }
      umma_commit(bar);
    }
    if (!mbar_wait(bar, phase)) {
      report_error(p.err, kDevErrTimeout);
      *abort_flag = 1;
    }
    phase ^= 1;
    tc_fence_after();
    __syncthreads();
    if (*abort_flag) {
      ok = false;
      break;
    }
  }

  // ---- epilogue: O / l -> bf16, LSE (TMEM load by the whole warp, stores for valid rows) ----
  if (ok) {
    uint32_t o[D];
#pragma unroll
    for (int c = 0; c < D / 32; ++c) tmem_ld32(tmem + lane_base + Cfg::kColO + 32 * c, o + 32 * c);
    tmem_ld_wait();
    reg_fence<D>(o);
    if (i_row < T) {
      const float inv_l = 1.0f / l_run;
      uint4* dst = reinterpret_cast<uint4*>(p.out + head_base + static_cast<size_t>(i_row) * row_stride);
#pragma unroll
      for (int ch = 0; ch < D / 8; ++ch) {
        uint4 u;
        u.x = pack_bf16x2(__uint_as_float(o[ch * 8 + 0]) * inv_l, __uint_as_float(o[ch * 8 + 1]) * inv_l);
        u.y = pack_bf16x2(__uint_as_float(o[ch * 8 + 2]) * inv_l, __uint_as_float(o[ch * 8 + 3]) * inv_l);
        u.z = pack_bf16x2(__uint_as_float(o[ch * 8 + 4]) * inv_l, __uint_as_float(o[ch * 8 + 5]) * inv_l);
        u.w = pack_bf16x2(__uint_as_float(o[ch * 8 + 6]) * inv_l, __uint_as_float(o[ch * 8 + 7]) * inv_l);
        dst[ch] = u;
      }
      if (p.lse != nullptr)
        p.lse[(static_cast<size_t>(b) * p.H + h) * T + i_row] = (m_run + __log2f(l_run)) * 0.69314718055994531f;
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
