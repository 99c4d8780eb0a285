// Host side of include/polar.h: argument checks, tensor maps and the launches of the normalisation
// and of the three GEMMs of every Polar Express step.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>
#include <mutex>

#include "attn.h"
#include "attn_internal.h"
#include "polar.cuh"
#include "polar.h"

namespace {

// The listing's polar_express_coeffs (a, b, c) per step: the method's definition, kept as data.
constexpr float kCoeffs[5][3] = {
    {8.156554524902461f, -22.48329292557795f, 15.878769915207462f},
    {4.042929935166739f, -2.808917465908714f, 0.5000178451051316f},
    {3.8916678022926607f, -2.772484153217685f, 0.5060648178503393f},
    {3.285753657755655f, -2.3681294933425376f, 0.46449024233003106f},
    {2.3465413258596377f, -1.7097828382687081f, 0.42323551169305323f},
};

size_t round256(size_t x) { return (x + 255) / 256 * 256; }

// The normalisation's chunk: 16384 elements, or more so that a matrix has at most 1024 chunks (the
// second pass sums a matrix's partial sums in every CTA).
int norm_chunk(long long mn) {
  long long c = 16384;
  while ((mn + c - 1) / c > 1024) c *= 2;
  return static_cast<int>(c);
}

struct PeLayout {
  size_t a, b, x, part, total;
  int chunk, nchunks;
};

PeLayout pe_layout(int batch, int m, int n) {
  const size_t s = static_cast<size_t>(m < n ? m : n);
  const long long mn = static_cast<long long>(m) * n;
  PeLayout l;
  l.chunk = norm_chunk(mn);
  l.nchunks = static_cast<int>((mn + l.chunk - 1) / l.chunk);
  l.a = 0;
  l.b = round256(static_cast<size_t>(batch) * s * s * 2);
  l.x = l.b + round256(static_cast<size_t>(batch) * s * s * 2);
  l.part = l.x + round256(static_cast<size_t>(batch) * m * n * 2);
  l.total = l.part + round256(static_cast<size_t>(batch) * l.nchunks * 4);
  return l;
}

// Both passes of the normalisation; `part` is the workspace's partial-sum region.
cudaError_t launch_normalize(cudaStream_t st, const void* G, void* X, int batch, int m, int n, uint8_t* ws) {
  const PeLayout l = pe_layout(batch, m, n);
  const long long mn = static_cast<long long>(m) * n;
  float* part = reinterpret_cast<float*>(ws + l.part);
  const dim3 grid(l.nchunks, batch);
  swa::frob_partial_kernel<<<grid, 256, 0, st>>>(static_cast<const __nv_bfloat16*>(G), part, mn, l.chunk);
  swa::frob_scale_kernel<<<grid, 256, 0, st>>>(static_cast<const __nv_bfloat16*>(G), static_cast<__nv_bfloat16*>(X),
                                               part, mn, l.chunk);
  return cudaGetLastError();
}

bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool overlap(const void* a, size_t na, const void* b, size_t nb) {
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
  return a0 < b0 + nb && b0 < a0 + na;
}

int check_shape(int batch, int m, int n) {
  if (batch < 1 || m < 8 || n < 8 || m % 8 != 0 || n % 8 != 0) return ATTN_ERR_INVALID_ARG;
  if (static_cast<long long>(batch) * m * n >= (1LL << 31)) return ATTN_ERR_INVALID_ARG;
  return ATTN_OK;
}

// A row-major [batch, rows, inner] bf16 matrix as a 3-D tensor map. K-major operand views take
// 128 rows x 64 inner elements per box; MN-major views 64 K rows x 64 inner (M / N) elements.
CUresult encode3d(PFN_cuTensorMapEncodeTiled_v12000 encode, CUtensorMap* map, const void* base, int batch, int rows,
                  int inner, bool mn_box) {
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(rows),
                              static_cast<cuuint64_t>(batch)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(inner) * 2, static_cast<cuuint64_t>(rows) * inner * 2};
  const cuuint32_t box[3] = {64, mn_box ? 64u : 128u, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

std::mutex g_pe_mu;
int g_pe_device = -1;

template <int A, int B, int BN>
cudaError_t set_attr_one() {
  return cudaFuncSetAttribute(swa::gemm_kernel<A, B, BN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              swa::GemmCfg<BN>::kSmemBytes);
}

using swa::kOpK;
using swa::kOpMN;
using swa::kOpSym;

cudaError_t set_attrs() {
  const cudaError_t e[10] = {set_attr_one<kOpK, kOpK, 128>(),     set_attr_one<kOpK, kOpK, 256>(),
                             set_attr_one<kOpMN, kOpMN, 128>(),   set_attr_one<kOpMN, kOpMN, 256>(),
                             set_attr_one<kOpSym, kOpSym, 128>(), set_attr_one<kOpSym, kOpSym, 256>(),
                             set_attr_one<kOpSym, kOpMN, 128>(),  set_attr_one<kOpSym, kOpMN, 256>(),
                             set_attr_one<kOpK, kOpSym, 128>(),   set_attr_one<kOpK, kOpSym, 256>()};
  for (cudaError_t x : e)
    if (x != cudaSuccess) return x;
  return cudaSuccess;
}

template <int A, int B>
void launch_gemm(int bn, int grid, cudaStream_t st, const swa::GemmParams& gp, const swa::GemmMaps& maps) {
  if (bn == 256)
    swa::gemm_kernel<A, B, 256><<<grid, 192, swa::GemmCfg<256>::kSmemBytes, st>>>(gp, maps);
  else
    swa::gemm_kernel<A, B, 128><<<grid, 192, swa::GemmCfg<128>::kSmemBytes, st>>>(gp, maps);
}

// Output tiles of one M x N matrix with BN-wide tiles (a symmetric output: those reaching the
// diagonal block or above it, as the kernel counts them).
long long tiles_per_mat(int M, int N, int bn, bool sym) {
  const long long tm = (M + 127) / 128, tn = (N + bn - 1) / bn;
  if (!sym) return tm * tn;
  long long c = 0;
  for (long long mt = 0; mt < tm; ++mt) c += tn - (128 * mt) / bn;
  return c;
}

// Output tile width: the one whose tiles finish in fewer rounds of the grid, counted in 128-column
// units of MMA work; 256 on a tie (it reads fewer operand bytes per product).
int choose_bn(int batch, int M, int N, bool sym, int sms, int* grid) {
  const long long t128 = tiles_per_mat(M, N, 128, sym) * batch, t256 = tiles_per_mat(M, N, 256, sym) * batch;
  const long long c128 = (t128 + sms - 1) / sms, c256 = 2 * ((t256 + sms - 1) / sms);
  const bool wide = c256 <= c128;
  const long long tiles = wide ? t256 : t128;
  *grid = static_cast<int>(tiles < sms ? tiles : sms);
  return wide ? 256 : 128;
}

// FLOPs the tensor cores execute for one GEMM launch: 2 K per in-range output element of the tiles
// it computes (for a symmetric output, the tiles reaching the diagonal block or above it).
double executed_flops(int batch, int M, int N, int K, bool sym, int sms) {
  int grid = 0;
  const int bn = choose_bn(batch, M, N, sym, sms, &grid);
  const int tm = (M + 127) / 128, tn = (N + bn - 1) / bn;
  double elems = 0.0;
  for (int mt = 0; mt < tm; ++mt)
    for (int nt = sym ? (128 * mt) / bn : 0; nt < tn; ++nt) {
      const int rows = M - 128 * mt < 128 ? M - 128 * mt : 128;
      const int cols = N - bn * nt < bn ? N - bn * nt : bn;
      elems += static_cast<double>(rows) * cols;
    }
  return 2.0 * K * elems * batch;
}

// D = alpha * P Q + beta * R over a batch; P is M x K, Q is K x N. Operand modes (swa::GemmOperand):
// P stored as [M, K] (kOpK), as [K, M] (kOpMN), or symmetric upper-block storage (kOpSym, M = K);
// Q stored as [N, K] (kOpK), as [K, N] (kOpMN), or symmetric (kOpSym, K = N). sym_out: D is symmetric
// and only its tiles on and above the diagonal are written.
int gemm(const swa_host::LibCtx& ctx, cudaStream_t st, int batch, int M, int N, int K, const void* P, int p_mode,
         const void* Q, int q_mode, float alpha, float beta, const void* R, void* D, bool sym_out) {
  swa::GemmMaps maps;
  std::memset(&maps, 0, sizeof(maps));
  // K-major view of P: [M rows, K inner]; MN-major view: [K rows, M inner] (equal shapes when symmetric)
  if (p_mode != kOpMN && encode3d(ctx.encode, &maps.pk, P, batch, M, K, false) != CUDA_SUCCESS) return ATTN_ERR_CUDA;
  if (p_mode != kOpK && encode3d(ctx.encode, &maps.pm, P, batch, K, M, true) != CUDA_SUCCESS) return ATTN_ERR_CUDA;
  if (q_mode != kOpMN && encode3d(ctx.encode, &maps.qk, Q, batch, N, K, false) != CUDA_SUCCESS) return ATTN_ERR_CUDA;
  if (q_mode != kOpK && encode3d(ctx.encode, &maps.qm, Q, batch, K, N, true) != CUDA_SUCCESS) return ATTN_ERR_CUDA;
  if (encode3d(ctx.encode, &maps.d, D, batch, M, N, false) != CUDA_SUCCESS) return ATTN_ERR_CUDA;
  swa::GemmParams gp{};
  gp.batch = batch;
  gp.M = M;
  gp.N = N;
  gp.K = K;
  gp.alpha = alpha;
  gp.beta = beta;
  gp.R = static_cast<const __nv_bfloat16*>(R);
  gp.err = ctx.d_err;
  gp.sym_out = sym_out ? 1 : 0;
  int grid = 0;
  const int bn = choose_bn(batch, M, N, sym_out, ctx.sm_count, &grid);
  if (p_mode == kOpK && q_mode == kOpK) launch_gemm<kOpK, kOpK>(bn, grid, st, gp, maps);
  else if (p_mode == kOpMN && q_mode == kOpMN) launch_gemm<kOpMN, kOpMN>(bn, grid, st, gp, maps);
  else if (p_mode == kOpSym && q_mode == kOpSym) launch_gemm<kOpSym, kOpSym>(bn, grid, st, gp, maps);
  else if (p_mode == kOpSym && q_mode == kOpMN) launch_gemm<kOpSym, kOpMN>(bn, grid, st, gp, maps);
  else if (p_mode == kOpK && q_mode == kOpSym) launch_gemm<kOpK, kOpSym>(bn, grid, st, gp, maps);
  else return ATTN_ERR_UNSUPPORTED;
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

int ensure_attrs(const swa_host::LibCtx& ctx) {
  std::lock_guard<std::mutex> g(g_pe_mu);
  if (g_pe_device == ctx.device) return ATTN_OK;
  if (swa_host::on_device(ctx.device, [] { return set_attrs(); }) != cudaSuccess) {
    cudaGetLastError();
    return ATTN_ERR_CUDA;
  }
  g_pe_device = ctx.device;
  return ATTN_OK;
}

// One step inside the library lock.
int step_locked(const swa_host::LibCtx& ctx, cudaStream_t st, const void* X, void* Y, int batch, int m, int n,
                int step, uint8_t* ws) {
  const PeLayout l = pe_layout(batch, m, n);
  void* A = ws + l.a;
  void* B = ws + l.b;
  const float a = kCoeffs[step][0], b = kCoeffs[step][1], c = kCoeffs[step][2];
  int rc;
  // A and B are symmetric: only their 128 x 128 blocks on and above the diagonal are computed and
  // stored, and the products that read them take each block below the diagonal as its mirror's
  // transpose.
  if (m <= n) {
    // wide: A = X X^T (m x m, K = n); B = c A A + b A; Y = a X + B X
    if ((rc = gemm(ctx, st, batch, m, m, n, X, kOpK, X, kOpK, 1.f, 0.f, nullptr, A, true)) != ATTN_OK) return rc;
    if ((rc = gemm(ctx, st, batch, m, m, m, A, kOpSym, A, kOpSym, c, b, A, B, true)) != ATTN_OK) return rc;
    return gemm(ctx, st, batch, m, n, m, B, kOpSym, X, kOpMN, 1.f, a, X, Y, false);
  }
  // tall: A = X^T X (n x n, K = m); B = c A A + b A; Y = a X + X B
  if ((rc = gemm(ctx, st, batch, n, n, m, X, kOpMN, X, kOpMN, 1.f, 0.f, nullptr, A, true)) != ATTN_OK) return rc;
  if ((rc = gemm(ctx, st, batch, n, n, n, A, kOpSym, A, kOpSym, c, b, A, B, true)) != ATTN_OK) return rc;
  return gemm(ctx, st, batch, m, n, n, X, kOpK, B, kOpSym, 1.f, a, X, Y, false);
}

}  // namespace

extern "C" {

double pe_step_flops(int batch, int m, int n) {
  if (check_shape(batch, m, n) != ATTN_OK) return 0.0;
  int sms = 0;
  const int dev_rc = swa_host::locked([&](const swa_host::LibCtx& ctx) -> int {
    sms = ctx.sm_count;
    return ATTN_OK;
  });
  if (dev_rc != ATTN_OK || sms <= 0) return 0.0;
  const int s = m < n ? m : n, l = m < n ? n : m;
  // A = X X^T (or X^T X), B = c A A + b A (both symmetric), Y = a X + B X (or X B)
  return executed_flops(batch, s, s, l, true, sms) + executed_flops(batch, s, s, s, true, sms) +
         executed_flops(batch, m, n, s, false, sms);
}

size_t pe_workspace_bytes(int batch, int m, int n) {
  if (batch < 1 || m < 1 || n < 1) return 0;
  return pe_layout(batch, m, n).total;
}

int pe_normalize(const void* G, void* X, int batch, int m, int n, void* workspace, size_t workspace_bytes,
                 void* stream) {
  int rc;
  if ((rc = check_shape(batch, m, n)) != ATTN_OK) return rc;
  if (!G || !X || !workspace || !al16(G) || !al16(X) || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return ATTN_ERR_INVALID_ARG;
  const PeLayout l = pe_layout(batch, m, n);
  if (workspace_bytes < l.total) return ATTN_ERR_INVALID_ARG;
  const size_t xb = static_cast<size_t>(batch) * m * n * 2;
  if ((G != X && overlap(G, xb, X, xb)) || overlap(X, xb, workspace, l.total) || overlap(G, xb, workspace, l.total))
    return ATTN_ERR_INVALID_ARG;
  return swa_host::locked([&](const swa_host::LibCtx& ctx) -> int {
    const cudaError_t e = swa_host::on_device(ctx.device, [&]() -> cudaError_t {
      return launch_normalize(static_cast<cudaStream_t>(stream), G, X, batch, m, n, static_cast<uint8_t*>(workspace));
    });
    return e != cudaSuccess ? ATTN_ERR_CUDA : ATTN_OK;
  });
}

int pe_step(const void* X, void* Y, int batch, int m, int n, int step, void* workspace, size_t workspace_bytes,
            void* stream) {
  int rc;
  if ((rc = check_shape(batch, m, n)) != ATTN_OK) return rc;
  if (step < 0 || step > 4) return ATTN_ERR_INVALID_ARG;
  if (!X || !Y || !workspace || !al16(X) || !al16(Y) || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return ATTN_ERR_INVALID_ARG;
  const PeLayout l = pe_layout(batch, m, n);
  if (workspace_bytes < l.total) return ATTN_ERR_INVALID_ARG;
  const size_t xb = static_cast<size_t>(batch) * m * n * 2;
  if (overlap(X, xb, Y, xb) || overlap(X, xb, workspace, l.total) || overlap(Y, xb, workspace, l.total))
    return ATTN_ERR_INVALID_ARG;
  return swa_host::locked([&](const swa_host::LibCtx& ctx) -> int {
    int r = ensure_attrs(ctx);
    if (r != ATTN_OK) return r;
    const cudaError_t e = swa_host::on_device(ctx.device, [&]() -> cudaError_t {
      r = step_locked(ctx, static_cast<cudaStream_t>(stream), X, Y, batch, m, n, step,
                      static_cast<uint8_t*>(workspace));
      return cudaSuccess;
    });
    return e != cudaSuccess ? ATTN_ERR_CUDA : r;
  });
}

int polar_express(const void* G, void* X, int batch, int m, int n, int steps, void* workspace,
                  size_t workspace_bytes, void* stream) {
  int rc;
  if ((rc = check_shape(batch, m, n)) != ATTN_OK) return rc;
  if (steps < 0 || steps > 5) return ATTN_ERR_INVALID_ARG;
  if (!G || !X || !workspace || !al16(G) || !al16(X) || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return ATTN_ERR_INVALID_ARG;
  const PeLayout l = pe_layout(batch, m, n);
  if (workspace_bytes < l.total) return ATTN_ERR_INVALID_ARG;
  const size_t xb = static_cast<size_t>(batch) * m * n * 2;
  if (overlap(G, xb, X, xb) || overlap(X, xb, workspace, l.total) || overlap(G, xb, workspace, l.total))
    return ATTN_ERR_INVALID_ARG;
  return swa_host::locked([&](const swa_host::LibCtx& ctx) -> int {
    int r = ensure_attrs(ctx);
    if (r != ATTN_OK) return r;
    const cudaError_t e = swa_host::on_device(ctx.device, [&]() -> cudaError_t {
      cudaStream_t st = static_cast<cudaStream_t>(stream);
      uint8_t* ws = static_cast<uint8_t*>(workspace);
      // the step sequence ping-pongs between X and the workspace's matrix so that it ends in X
      void* bufs[2] = {X, ws + l.x};
      int cur = steps % 2 == 0 ? 0 : 1;
      if (launch_normalize(st, G, bufs[cur], batch, m, n, ws) != cudaSuccess) {
        r = ATTN_ERR_CUDA;
        return cudaSuccess;
      }
      for (int s = 0; s < steps && r == ATTN_OK; ++s) {
        r = step_locked(ctx, st, bufs[cur], bufs[cur ^ 1], batch, m, n, s, ws);
        cur ^= 1;
      }
      return cudaSuccess;
    });
    return e != cudaSuccess ? ATTN_ERR_CUDA : r;
  });
}

}  // extern "C"
