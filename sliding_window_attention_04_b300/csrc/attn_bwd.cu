// Host side of the attention backward entry points declared in include/attn.h: argument
// validation, the workspace layout, tensor maps and the three launches on the caller's stream.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "attn.h"
#include "attn_bwd.cuh"
#include "attn_bwd_ws.cuh"
#include "attn_internal.h"

namespace {

constexpr size_t kAlign = 256;

size_t round_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

// Workspace layout: q^ bf16 [B, T, H, D] | k^ bf16 [B, T, Hkv, D] | delta fp32 [B, H, Tp] |
// -lse log2(e) fp32 [B, H, Tp] | dq^ fp32 [B, T, H, D] | ticket counter (int), each part starting on
// a 256-byte boundary; Tp = T rounded up to a multiple of 128 (rows of whole query tiles, for
// 512-byte bulk copies).
struct WsLayout {
  size_t qh, kh, delta, nlse, dqh, tickets, total;
};

WsLayout layout(int B, int H, int Hkv, int T, int D) {
  const size_t nq = static_cast<size_t>(B) * T * H * D, nk = static_cast<size_t>(B) * T * Hkv * D;
  const size_t Tp = (static_cast<size_t>(T) + swa::kTile - 1) / swa::kTile * swa::kTile;
  WsLayout l;
  l.qh = 0;
  l.kh = round_up(l.qh + nq * 2);
  l.delta = round_up(l.kh + nk * 2);
  l.nlse = round_up(l.delta + static_cast<size_t>(B) * H * Tp * 4);
  l.dqh = round_up(l.nlse + static_cast<size_t>(B) * H * Tp * 4);
  l.tickets = round_up(l.dqh + nq * 4);
  l.total = l.tickets + kAlign;
  return l;
}

// 4-D (d, h, t, b) view of an fp32 [B, T, H, D] tensor, boxes of 128 rows x 32 columns (128 bytes)
// with the 128-byte swizzle; rows past T are dropped by stores and reductions.
CUresult encode_f32_map(PFN_cuTensorMapEncodeTiled_v12000 encode, CUtensorMap* map, const void* base, int B, int H,
                        int T, int D) {
  const cuuint64_t dims[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(T),
                              static_cast<cuuint64_t>(B)};
  const cuuint64_t strides[3] = {static_cast<cuuint64_t>(D) * 4, static_cast<cuuint64_t>(H) * D * 4,
                                 static_cast<cuuint64_t>(T) * H * D * 4};
  const cuuint32_t box[4] = {32, 1, static_cast<cuuint32_t>(swa::kTile), 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  return encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, const_cast<void*>(base), dims, strides, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
  return a0 < b0 + nb && b0 < a0 + na;
}

std::mutex g_attr_mu;
int g_attr_device = -1;  // device whose kernel attributes have been set

// Resident CTAs per SM of the prep and finalize passes (by their shared-memory rings and registers),
// indexed by D / 64 (D = 32, 64, 128 -> 0, 1, 2); set with the attributes.
int g_prep_ctas_per_sm[3] = {1, 1, 1};
int g_fin_ctas_per_sm[3] = {1, 1, 1};

template <int D>
cudaError_t set_bwd_attrs() {
  cudaError_t e = cudaFuncSetAttribute(swa::attn_bwd_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       swa::BwdCfg<D>::kSmemBytes);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(swa::attn_bwd_prep_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           swa::PrepCfg<D>::kSmemBytes);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(swa::attn_bwd_dq_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           swa::FinCfg<D>::kSmemBytes);
  if (e != cudaSuccess) return e;
  int n = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, swa::attn_bwd_prep_kernel<D>, 256, swa::PrepCfg<D>::kSmemBytes);
  if (e != cudaSuccess) return e;
  if (n < 1) return cudaErrorInvalidConfiguration;
  g_prep_ctas_per_sm[D / 64] = n;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, swa::attn_bwd_dq_kernel<D>, 256, swa::FinCfg<D>::kSmemBytes);
  if (e != cudaSuccess) return e;
  if (n < 1) return cudaErrorInvalidConfiguration;
  g_fin_ctas_per_sm[D / 64] = n;
  if (D == 128) return e;
  return cudaFuncSetAttribute(swa::attn_bwd_ws_kernel<D == 128 ? 64 : D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              swa::BwdWsCfg<D == 128 ? 64 : D>::kSmemBytes);
}

template <int D>
int launch_bwd(const swa::BwdParams& p, const swa_host::LibCtx& ctx, cudaStream_t st) {
  swa::BwdMaps maps;
  if (swa_host::encode_bf16_tile_map(ctx.encode, &maps.qh, p.qh, p.B, p.H, p.T, D) != CUDA_SUCCESS ||
      swa_host::encode_bf16_tile_map(ctx.encode, &maps.kh, p.kh, p.B, p.Hkv, p.T, D) != CUDA_SUCCESS ||
      swa_host::encode_bf16_tile_map(ctx.encode, &maps.v, p.v, p.B, p.Hkv, p.T, D) != CUDA_SUCCESS ||
      swa_host::encode_bf16_tile_map(ctx.encode, &maps.dout, p.dout, p.B, p.H, p.T, D) != CUDA_SUCCESS ||
      encode_f32_map(ctx.encode, &maps.dqh, p.dqh, p.B, p.H, p.T, D) != CUDA_SUCCESS ||
      encode_f32_map(ctx.encode, &maps.dk, p.dk, p.B, p.Hkv, p.T, D) != CUDA_SUCCESS ||
      encode_f32_map(ctx.encode, &maps.dv, p.dv, p.B, p.Hkv, p.T, D) != CUDA_SUCCESS)
    return ATTN_ERR_CUDA;
  // prep and finalize: one group of rows per warp step, eight warps per CTA, as many CTAs as stay
  // resident (each warp then strides over the groups)
  const long long nq = static_cast<long long>(p.B) * p.T * p.H, nk = static_cast<long long>(p.B) * p.T * p.Hkv;
  using PC = swa::PrepCfg<D>;
  using FC = swa::FinCfg<D>;
  const long long prep_groups = (nq + PC::kQRows - 1) / PC::kQRows + (nk + PC::kKRows - 1) / PC::kKRows;
  const long long prep_cap = static_cast<long long>(g_prep_ctas_per_sm[D / 64]) * ctx.sm_count;
  const long long prep_need = (prep_groups + PC::kWarps - 1) / PC::kWarps;
  const int prep_grid = static_cast<int>(prep_need < prep_cap ? prep_need : prep_cap);
  swa::attn_bwd_prep_kernel<D><<<prep_grid, PC::kWarps * 32, PC::kSmemBytes, st>>>(p);
  const long long ctas = static_cast<long long>(p.B) * p.Hkv * p.n_ktiles;
  if constexpr (D <= 64) {
    // persistent warp-specialised pipeline: one CTA per SM takes key tiles from the ticket counter
    if (ctas >= (1LL << 31)) return ATTN_ERR_INVALID_ARG;
    const int grid = static_cast<int>(ctas < ctx.sm_count ? ctas : ctx.sm_count);
    swa::attn_bwd_ws_kernel<D><<<grid, swa::BwdWsCfg<D>::kThreads, swa::BwdWsCfg<D>::kSmemBytes, st>>>(
        p, maps, p.tickets, static_cast<int>(ctas));
  } else {
    swa::attn_bwd_kernel<D><<<static_cast<unsigned>(ctas), swa::BwdCfg<D>::kThreads, swa::BwdCfg<D>::kSmemBytes,
                              st>>>(p, maps);
  }
  const long long fin_groups = (nq + FC::kRows - 1) / FC::kRows + (nk + FC::kRows - 1) / FC::kRows;
  const long long fin_cap = static_cast<long long>(g_fin_ctas_per_sm[D / 64]) * ctx.sm_count;
  const long long fin_need = (fin_groups + FC::kWarps - 1) / FC::kWarps;
  const int fin_grid = static_cast<int>(fin_need < fin_cap ? fin_need : fin_cap);
  swa::attn_bwd_dq_kernel<D><<<fin_grid, FC::kWarps * 32, FC::kSmemBytes, st>>>(p);
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

}  // namespace

extern "C" {

size_t attn_bwd_workspace_bytes(int B, int H, int H_kv, int T, int D) {
  if (B < 1 || H < 1 || H_kv < 1 || T < 1 || D < 1) return 0;
  return layout(B, H, H_kv, T, D).total;
}

int attn_bwd(const void* q, const void* k, const void* v, const void* out, const float* lse, const void* dout,
             float* dq, float* dk, float* dv, void* workspace, size_t workspace_bytes, int B, int H, int H_kv, int T,
             int D, int window, int causal, float rope_base, float eps, void* stream) {
  // ---- argument checks (host only, nothing launched) ----
  if (!q || !k || !v || !out || !lse || !dout || !dq || !dk || !dv || !workspace) return ATTN_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16) || !aligned(dout, 16) ||
      !aligned(dq, 16) || !aligned(dk, 16) || !aligned(dv, 16) || !aligned(lse, 4) || !aligned(workspace, kAlign))
    return ATTN_ERR_INVALID_ARG;
  if (B < 1 || H < 1 || T < 1 || D < 1) return ATTN_ERR_INVALID_ARG;
  if (H_kv < 1 || H_kv > H || H % H_kv != 0) return ATTN_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return ATTN_ERR_INVALID_ARG;
  if (!std::isfinite(rope_base) || rope_base < 0.f) return ATTN_ERR_INVALID_ARG;
  if (std::isnan(eps) || std::isinf(eps)) return ATTN_ERR_INVALID_ARG;
  const long long n_elem = static_cast<long long>(B) * T * H * D;
  if (n_elem >= (1LL << 31)) return ATTN_ERR_INVALID_ARG;
  if (D != 32 && D != 64 && D != 128) return ATTN_ERR_UNSUPPORTED;
  const WsLayout l = layout(B, H, H_kv, T, D);
  if (workspace_bytes < l.total) return ATTN_ERR_INVALID_ARG;
  const size_t qb = static_cast<size_t>(n_elem) * 2, kb = qb / static_cast<size_t>(H / H_kv);
  const size_t lb = static_cast<size_t>(B) * H * T * 4;
  // outputs must not overlap an input, each other or the workspace
  const void* ins[6] = {q, k, v, out, lse, dout};
  const size_t in_bytes[6] = {qb, kb, kb, qb, lb, qb};
  const void* outs[4] = {dq, dk, dv, workspace};
  const size_t out_bytes[4] = {qb * 2, kb * 2, kb * 2, l.total};
  for (int a = 0; a < 4; ++a) {
    for (int i = 0; i < 6; ++i)
      if (overlaps(outs[a], out_bytes[a], ins[i], in_bytes[i])) return ATTN_ERR_INVALID_ARG;
    for (int c = a + 1; c < 4; ++c)
      if (overlaps(outs[a], out_bytes[a], outs[c], out_bytes[c])) return ATTN_ERR_INVALID_ARG;
  }

  return swa_host::locked([&](const swa_host::LibCtx& ctx) -> int {
    {
      std::lock_guard<std::mutex> g(g_attr_mu);
      if (g_attr_device != ctx.device) {
        const cudaError_t e = swa_host::on_device(ctx.device, [] {
          cudaError_t r;
          if ((r = set_bwd_attrs<32>()) != cudaSuccess) return r;
          if ((r = set_bwd_attrs<64>()) != cudaSuccess) return r;
          return set_bwd_attrs<128>();
        });
        if (e != cudaSuccess) {
          cudaGetLastError();
          return ATTN_ERR_CUDA;
        }
        g_attr_device = ctx.device;
      }
    }
    const float4* table = nullptr;
    const float4* rows = nullptr;
    int table_T = 0;
    if (rope_base > 0.f && swa_host::rope_table_locked(D, rope_base, T, &table, &table_T, &rows) != ATTN_OK)
      return ATTN_ERR_CUDA;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    swa::BwdParams p{};
    p.q = static_cast<const __nv_bfloat16*>(q);
    p.k = static_cast<const __nv_bfloat16*>(k);
    p.v = static_cast<const __nv_bfloat16*>(v);
    p.out = static_cast<const __nv_bfloat16*>(out);
    p.lse = lse;
    p.dout = static_cast<const __nv_bfloat16*>(dout);
    p.dq = dq;
    p.dk = dk;
    p.dv = dv;
    p.qh = reinterpret_cast<__nv_bfloat16*>(ws + l.qh);
    p.kh = reinterpret_cast<__nv_bfloat16*>(ws + l.kh);
    p.delta = reinterpret_cast<float*>(ws + l.delta);
    p.nlse = reinterpret_cast<float*>(ws + l.nlse);
    p.tickets = reinterpret_cast<int*>(ws + l.tickets);
    p.dqh = reinterpret_cast<float*>(ws + l.dqh);
    p.rope = rows;
    p.err = ctx.d_err;
    p.B = B;
    p.H = H;
    p.Hkv = H_kv;
    p.kv_group = H / H_kv;
    p.T = T;
    p.window = window < 0 ? -1 : window;
    p.causal = causal;
    p.use_norm = eps >= 0.f ? 1 : 0;
    p.eps = eps >= 0.f ? eps : 0.f;
    p.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(D)));
    p.scale = static_cast<float>(1.0 / std::sqrt(static_cast<double>(D)));
    p.n_ktiles = (T + swa::kTile - 1) / swa::kTile;
    p.Tp = p.n_ktiles * swa::kTile;
    if (static_cast<long long>(B) * H_kv * p.n_ktiles >= (1LL << 31)) return ATTN_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int rc = ATTN_OK;
    const cudaError_t e = swa_host::on_device(ctx.device, [&]() -> cudaError_t {
      switch (D) {
        case 32: rc = launch_bwd<32>(p, ctx, st); break;
        case 64: rc = launch_bwd<64>(p, ctx, st); break;
        default: rc = launch_bwd<128>(p, ctx, st); break;
      }
      return cudaSuccess;
    });
    if (e != cudaSuccess) return ATTN_ERR_CUDA;
    return rc;
  });
}

}  // extern "C"
