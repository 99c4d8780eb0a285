// Host side of the C ABI declared in include/attn.h: argument validation, the cached cos/sin
// tables, the device error word and kernel launches on the caller's stream.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdint>
#include <cstdio>
#include <map>
#include <mutex>
#include <utility>
#include <vector>

#include "attn.h"
#include "attn_internal.h"
#include "attn_fwd_simple.cuh"
#include "attn_fwd_ws.cuh"

namespace {

struct RopeTable {
  float4* ptr = nullptr;
  int T = 0;  // positions covered (the table's row stride)
};

// Ticket counters of the persistent kernel: one (ticket, exits) pair per slot, 128 bytes apart.
// Each call takes a slot; the kernel's last CTA resets its pair to zero on exit. Calls made outside
// stream capture take the next slot of the first kSchedSlots / 2, round robin, and a slot is only
// ever reused after its previous kernel has finished: on the same stream by stream order, on another
// stream because the new call's stream first waits for an event recorded after the previous kernel
// of that slot (so more calls in flight than slots are serialised, never corrupted). Calls made
// while the stream is being captured into a CUDA graph take the next slot of the other half; they
// cannot wait for work outside the capture, so graph launches that run at the same time must hold
// fewer captured calls than that half.
constexpr int kSchedSlots = 256;
constexpr int kSchedStride = 32;  // ints per slot

struct SchedSlot {
  cudaEvent_t done = nullptr;    // recorded on `stream` right after the slot's last launch
  cudaStream_t stream = nullptr;
  bool used = false;
};

// Tensor maps depend only on the base pointer and the shape; they are cached so that repeated calls
// on the same buffers skip the encoding.
struct MapKey {
  const void* base;
  int B, H, T, D, rows;
  bool operator<(const MapKey& o) const {
    if (base != o.base) return base < o.base;
    if (B != o.B) return B < o.B;
    if (H != o.H) return H < o.H;
    if (T != o.T) return T < o.T;
    if (D != o.D) return D < o.D;
    return rows < o.rows;
  }
};
constexpr size_t kMapCacheMax = 1024;

struct State {
  std::mutex mu;
  bool inited = false;
  int device = -1;
  int sm_count = 0;
  int* d_err = nullptr;
  int* d_sched = nullptr;
  unsigned sched_next = 0;    // next eager slot (first half)
  unsigned capture_next = 0;  // next slot of calls under stream capture (second half)
  SchedSlot slots[kSchedSlots];
  std::map<MapKey, CUtensorMap> maps;
  bool ws_ok[3] = {false, false, false};  // warp-specialised kernel usable for D = 32, 64, 128
  std::map<std::pair<int, float>, RopeTable> tables;  // (D, base) -> table
  std::vector<float4*> retired;                       // outgrown tables, freed at destroy
  PFN_cuTensorMapEncodeTiled_v12000 encode_tiled = nullptr;
};

State& state() {
  static State s;
  return s;
}

// Runs `f` with `dev` as the current device and restores the caller's device afterwards.
template <typename F>
cudaError_t with_device(int dev, F&& f) {
  int prev = -1;
  cudaError_t e = cudaGetDevice(&prev);
  if (e != cudaSuccess) return e;
  if (prev != dev && (e = cudaSetDevice(dev)) != cudaSuccess) return e;
  cudaError_t r = f();
  if (prev != dev) cudaSetDevice(prev);
  return r;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
  return a0 < b0 + nb && b0 < a0 + na;
}

template <int D>
cudaError_t set_kernel_attrs() {
  return cudaFuncSetAttribute(swa::attn_fwd_simple_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              swa::SimpleCfg<D>::kSmemBytes);
}

// The warp-specialised kernel re-divides its registers at run time (setmaxnreg); that split adds
// up to the registers of the launch only if the kernel was compiled to exactly kLaunchRegs per
// thread. With any other count the kernel is not used. Both instantiations (the general one and the
// one for calls with the QK-norm on and no gate) must pass.
template <int D, bool kCommon>
cudaError_t set_ws_attrs_one(bool* usable) {
  *usable = false;
  cudaFuncAttributes fa;
  cudaError_t e = cudaFuncGetAttributes(&fa, swa::attn_fwd_ws_kernel<D, kCommon>);
  if (e != cudaSuccess) return e;
  if (fa.numRegs != swa::WsCfg<D>::kLaunchRegs) return cudaSuccess;
  e = cudaFuncSetAttribute(swa::attn_fwd_ws_kernel<D, kCommon>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           swa::WsCfg<D>::kSmemBytes);
  if (e != cudaSuccess) return e;
  *usable = true;
  return cudaSuccess;
}

template <int D>
cudaError_t set_ws_attrs(bool* usable) {
  bool general = false, common = false;
  cudaError_t e = set_ws_attrs_one<D, false>(&general);
  if (e != cudaSuccess) return e;
  if ((e = set_ws_attrs_one<D, true>(&common)) != cudaSuccess) return e;
  *usable = general && common;
  return cudaSuccess;
}

// 4-D view (d, h, t, b) of a [B, T, H, D] bf16 tensor; one box is `rows` rows (a 128-row tile, or
// the 32 rows of one warp for the forward's output) of one head, in shared memory in the tensor
// core's swizzled layout (128-byte rows: 128-byte swizzle, 64-byte rows: 64-byte swizzle). Rows past
// T read as zero and are not written by stores.
CUresult encode_tile_map(PFN_cuTensorMapEncodeTiled_v12000 encode, CUtensorMap* map, const void* base, int B,
                         int H, int T, int D, int rows = swa::kTile) {
  const cuuint64_t dims[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(T),
                              static_cast<cuuint64_t>(B)};
  const cuuint64_t strides[3] = {static_cast<cuuint64_t>(D) * 2, static_cast<cuuint64_t>(H) * D * 2,
                                 static_cast<cuuint64_t>(T) * H * D * 2};
  // D = 128 rows are 256 bytes: a box covers 64 columns (the 128-byte swizzle span), two per tile
  const cuuint32_t box[4] = {static_cast<cuuint32_t>(D > 64 ? 64 : D), 1, static_cast<cuuint32_t>(rows), 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  return encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, D >= 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

// cos / sin of t * base^(-2i/D) for t < T, i < D/2, evaluated in double and rounded to fp32.
// Layout [D/4][T] of float4 (cos_2m, cos_2m+1, sin_2m, sin_2m+1): for a fixed pair group the
// positions are contiguous, so a warp whose threads hold consecutive rows loads whole lines.
// One allocation: [D/4][T] (entry m of position t at m T + t: consecutive positions side by side, as
// the forward's prologue reads a tile of rows), then the same entries [T][D/4] (at T D/4 + t D/4 + m:
// one position's entries side by side, as the backward's passes read them).
cudaError_t build_table(int D, float base, int T, float4** out) {
  const size_t n = static_cast<size_t>(T) * (D / 4);
  std::vector<float4> h(2 * n);
  for (int t = 0; t < T; ++t)
    for (int m = 0; m < D / 4; ++m) {
      float cs[4];
      for (int k = 0; k < 2; ++k) {
        const int i = 2 * m + k;
        const double theta = static_cast<double>(t) * std::pow(static_cast<double>(base), -2.0 * i / D);
        cs[2 * k] = static_cast<float>(std::cos(theta));
        cs[2 * k + 1] = static_cast<float>(std::sin(theta));
      }
      h[static_cast<size_t>(m) * T + t] = make_float4(cs[0], cs[2], cs[1], cs[3]);
      h[n + static_cast<size_t>(t) * (D / 4) + m] = make_float4(cs[0], cs[2], cs[1], cs[3]);
    }
  float4* d = nullptr;
  cudaError_t e = cudaMalloc(&d, h.size() * sizeof(float4));
  if (e != cudaSuccess) return e;
  e = cudaMemcpy(d, h.data(), h.size() * sizeof(float4), cudaMemcpyHostToDevice);
  if (e != cudaSuccess) {
    cudaFree(d);
    return e;
  }
  *out = d;
  return cudaSuccess;
}

// One CTA waits on an mbarrier that nothing arrives on; the bounded wait gives up and the
// kernel records the timeout in the error word, then returns.
__global__ void selftest_wait_timeout_kernel(int* err) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    swa::mbar_init(&bar, 1);
    swa::fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0 && !swa::mbar_wait(&bar, 0)) swa::report_error(err, swa::kDevErrTimeout);
}

template <int D>
cudaError_t launch_simple(const swa::AttnParams& p, cudaStream_t stream) {
  const int grid = p.B * p.H * p.n_qtiles;
  swa::attn_fwd_simple_kernel<D><<<grid, swa::SimpleCfg<D>::kThreads, swa::SimpleCfg<D>::kSmemBytes, stream>>>(p);
  return cudaGetLastError();
}

// The cached tensor map of a [B, T, H, D] bf16 tensor at `base` (encoded on first use).
const CUtensorMap* cached_map(std::map<MapKey, CUtensorMap>& cache, PFN_cuTensorMapEncodeTiled_v12000 encode,
                              const void* base, int B, int H, int T, int D, int rows = swa::kTile) {
  const MapKey key{base, B, H, T, D, rows};
  auto it = cache.find(key);
  if (it != cache.end()) return &it->second;
  CUtensorMap m;
  if (encode_tile_map(encode, &m, base, B, H, T, D, rows) != CUDA_SUCCESS) return nullptr;
  if (cache.size() >= kMapCacheMax) cache.clear();
  return &cache.emplace(key, m).first->second;
}

template <int D>
int launch_ws(const swa::AttnParams& p, std::map<MapKey, CUtensorMap>& cache,
              PFN_cuTensorMapEncodeTiled_v12000 encode, int sm_count, int* sched, cudaStream_t stream) {
  swa::WsMaps maps;
  const CUtensorMap* mq = cached_map(cache, encode, p.q, p.B, p.H, p.T, D);
  const CUtensorMap* mk = cached_map(cache, encode, p.k, p.B, p.Hkv, p.T, D);
  const CUtensorMap* mv = cached_map(cache, encode, p.v, p.B, p.Hkv, p.T, D);
  const CUtensorMap* mo = cached_map(cache, encode, p.out, p.B, p.H, p.T, D, swa::kOutRows);
  if (!mq || !mk || !mv || !mo) return ATTN_ERR_CUDA;
  maps.q = *mq;
  maps.k = *mk;
  maps.v = *mv;
  maps.out = *mo;
  // Work is handed out in chunks of 256-row query blocks of one head (see the kernel). Where
  // consecutive blocks of a head can share key tiles through the ring (causal, window at most the
  // ring's depth in key tiles), all but the last heads run as one chunk each (all their blocks, so
  // every K^ tile is loaded and transformed once or twice instead of up to three times); the last
  // heads, about two waves of tickets, run as pairs of blocks, heaviest first, which balances the
  // tail. Pairs take heads in groups whose K and V fit in half of L2 together.
  const long long n_qb = (p.T + 2 * swa::kTile - 1) / (2 * swa::kTile);
  const long long n_bh = static_cast<long long>(p.B) * p.H;
  const long long cpb = (n_qb + 1) / 2;  // pairs per head
  swa::AttnParams pk = p;
  const long long kv_head_bytes = 2LL * p.T * D * 2 / p.kv_group;  // K + V per query head (a group shares them)
  const long long hg = (64LL << 20) / kv_head_bytes;
  pk.head_group = static_cast<int>(hg < 1 ? 1 : (hg > (1 << 20) ? (1 << 20) : hg));
  const bool chains = p.causal && p.window >= 0 && p.window <= swa::WsCfg<D>::kStages * swa::kTile && n_qb > 1;
  const long long tail = 2 * ((sm_count + cpb - 1) / cpb);  // heads run as pairs
  pk.n_long = chains && n_bh > tail ? static_cast<int>(n_bh - tail) : 0;
  const long long chunks = pk.n_long + (n_bh - pk.n_long) * cpb;
  if (chunks >= (1LL << 31)) return ATTN_ERR_INVALID_ARG;
  const int grid = static_cast<int>(chunks < sm_count ? chunks : sm_count);
  // QK-norm on, no gate: the instantiation without the other modes' code
  const bool common = p.use_norm && p.ve == nullptr;
  if (common)
    swa::attn_fwd_ws_kernel<D, true><<<grid, swa::WsCfg<D>::kThreads, swa::WsCfg<D>::kSmemBytes, stream>>>(
        pk, maps, sched, static_cast<int>(chunks));
  else
    swa::attn_fwd_ws_kernel<D, false><<<grid, swa::WsCfg<D>::kThreads, swa::WsCfg<D>::kSmemBytes, stream>>>(
        pk, maps, sched, static_cast<int>(chunks));
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

// ---- allocation-free variant: everything it needs beyond the caller's tensors lives here ----
// Layout: bytes [0, 256) hold the device error word, then kNoAllocTablePairs (cos, sin) pairs.
constexpr size_t kNoAllocHeaderBytes = 256;
constexpr size_t kNoAllocTablePairs = size_t(1) << 19;  // T * D / 2 <= 524288 pairs (4 MiB)
constexpr size_t kNoAllocBytes = kNoAllocHeaderBytes + kNoAllocTablePairs * sizeof(float2);

// Fills the cos / sin table for (T, D, base) in the layout of build_table ([D/4][T] float4). Runs
// on the caller's stream right before the attention kernel. The error word is left alone: it
// keeps a timeout until attn_noalloc_status reads and clears it.
__global__ void noalloc_prepare_kernel(unsigned char* scratch, int T, int D, float base) {
  float* table = reinterpret_cast<float*>(scratch + kNoAllocHeaderBytes);
  const int half = D / 2;
  const size_t n = base > 0.f ? static_cast<size_t>(T) * half : 0;
  for (size_t idx = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; idx < n;
       idx += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const int t = static_cast<int>(idx / half), i = static_cast<int>(idx % half);
    const double theta = static_cast<double>(t) * pow(static_cast<double>(base), -2.0 * i / D);
    double sn, cs;
    sincos(theta, &sn, &cs);
    float* dst = table + 4 * (static_cast<size_t>(i / 2) * T + t) + (i % 2);
    dst[0] = static_cast<float>(cs);
    dst[2] = static_cast<float>(sn);
  }
}

struct NoAllocDevice {
  unsigned char* scratch = nullptr;  // device address of g_noalloc_scratch on that device
};

std::mutex& noalloc_mutex() {
  static std::mutex m;
  return m;
}

std::map<int, NoAllocDevice>& noalloc_devices() {
  static std::map<int, NoAllocDevice> m;
  return m;
}

}  // namespace

// The allocation-free entry point's scratch. In host code this name is only a stand-in for the
// device array; its device address comes from cudaGetSymbolAddress, once per device.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocBytes];

namespace {

// First use on the current device: check it, raise the kernels' shared-memory limits and look
// up the device address of the scratch array. Returns ATTN_OK or an error code.
int noalloc_setup(int* dev_out, unsigned char** scratch_out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return ATTN_ERR_NO_DEVICE;
  }
  std::lock_guard<std::mutex> lock(noalloc_mutex());
  auto it = noalloc_devices().find(dev);
  if (it == noalloc_devices().end()) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
      cudaGetLastError();
      return ATTN_ERR_CUDA;
    }
    if (major != 10 || minor != 3) return ATTN_ERR_NO_DEVICE;
    if (set_kernel_attrs<32>() != cudaSuccess || set_kernel_attrs<64>() != cudaSuccess ||
        set_kernel_attrs<128>() != cudaSuccess) {
      cudaGetLastError();
      return ATTN_ERR_CUDA;
    }
    unsigned char* ptr = nullptr;
    if (cudaGetSymbolAddress(reinterpret_cast<void**>(&ptr), g_noalloc_scratch) != cudaSuccess || ptr == nullptr) {
      cudaGetLastError();
      return ATTN_ERR_CUDA;
    }
    NoAllocDevice d;
    d.scratch = ptr;
    it = noalloc_devices().emplace(dev, d).first;
  }
  *dev_out = dev;
  *scratch_out = it->second.scratch;
  return ATTN_OK;
}

}  // namespace

namespace swa_host {

int locked(const std::function<int(const LibCtx&)>& f) {
  State& s = state();
  std::lock_guard<std::mutex> lock(s.mu);
  if (!s.inited) return ATTN_ERR_NOT_INITIALIZED;
  const LibCtx ctx{s.device, s.sm_count, s.d_err, s.encode_tiled};
  return f(ctx);
}

int rope_table_locked(int D, float base, int T, const float4** table, int* table_T, const float4** rows) {
  State& s = state();
  RopeTable& t = s.tables[std::make_pair(D, base)];
  if (t.T < T) {
    float4* fresh = nullptr;
    if (with_device(s.device, [&] { return build_table(D, base, T, &fresh); }) != cudaSuccess) return ATTN_ERR_CUDA;
    if (t.ptr) s.retired.push_back(t.ptr);
    t.ptr = fresh;
    t.T = T;
  }
  *table = t.ptr;
  *table_T = t.T;
  if (rows != nullptr) *rows = t.ptr + static_cast<size_t>(t.T) * (D / 4);
  return ATTN_OK;
}

CUresult encode_bf16_tile_map(PFN_cuTensorMapEncodeTiled_v12000 encode, CUtensorMap* map, const void* base, int B,
                              int H, int T, int D) {
  return encode_tile_map(encode, map, base, B, H, T, D);
}

cudaError_t on_device(int dev, const std::function<cudaError_t()>& f) { return with_device(dev, f); }

}  // namespace swa_host

extern "C" {

int attn_init(int device) {
  State& s = state();
  std::lock_guard<std::mutex> lock(s.mu);
  if (s.inited) return device == s.device ? ATTN_OK : ATTN_ERR_INVALID_ARG;
  int count = 0;
  if (cudaGetDeviceCount(&count) != cudaSuccess || count <= 0) {
    cudaGetLastError();
    return ATTN_ERR_NO_DEVICE;
  }
  if (device < 0 || device >= count) return ATTN_ERR_INVALID_ARG;
  cudaDeviceProp prop;
  if (cudaGetDeviceProperties(&prop, device) != cudaSuccess) return ATTN_ERR_CUDA;
  if (prop.major != 10 || prop.minor != 3) return ATTN_ERR_NO_DEVICE;
  int* d_err = nullptr;
  int* d_sched = nullptr;
  bool ws_ok[3] = {false, false, false};
  cudaError_t e = with_device(device, [&]() -> cudaError_t {
    cudaError_t r;
    if ((r = set_kernel_attrs<32>()) != cudaSuccess) return r;
    if ((r = set_kernel_attrs<64>()) != cudaSuccess) return r;
    if ((r = set_kernel_attrs<128>()) != cudaSuccess) return r;
    if ((r = set_ws_attrs<32>(&ws_ok[0])) != cudaSuccess) return r;
    if ((r = set_ws_attrs<64>(&ws_ok[1])) != cudaSuccess) return r;
    if ((r = set_ws_attrs<128>(&ws_ok[2])) != cudaSuccess) return r;
    if ((r = cudaMalloc(&d_err, sizeof(int))) != cudaSuccess) return r;
    if ((r = cudaMemset(d_err, 0, sizeof(int))) != cudaSuccess) return r;
    const size_t sched_bytes = sizeof(int) * kSchedSlots * kSchedStride;
    if ((r = cudaMalloc(&d_sched, sched_bytes)) != cudaSuccess) return r;
    if ((r = cudaMemset(d_sched, 0, sched_bytes)) != cudaSuccess) return r;
    for (int i = 0; i < kSchedSlots; ++i) {
      s.slots[i] = SchedSlot{};
      if ((r = cudaEventCreateWithFlags(&s.slots[i].done, cudaEventDisableTiming)) != cudaSuccess) return r;
    }
    return cudaDeviceSynchronize();
  });
  if (e != cudaSuccess) {
    cudaGetLastError();
    if (d_err) cudaFree(d_err);
    if (d_sched) cudaFree(d_sched);
    for (SchedSlot& sl : s.slots) {
      if (sl.done) cudaEventDestroy(sl.done);
      sl = SchedSlot{};
    }
    return ATTN_ERR_CUDA;
  }
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult qres;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &qres) !=
          cudaSuccess ||
      qres != cudaDriverEntryPointSuccess || fn == nullptr) {
    cudaGetLastError();
    with_device(device, [&]() -> cudaError_t {
      cudaFree(d_err);
      cudaFree(d_sched);
      for (SchedSlot& sl : s.slots) {
        if (sl.done) cudaEventDestroy(sl.done);
        sl = SchedSlot{};
      }
      return cudaSuccess;
    });
    return ATTN_ERR_CUDA;
  }
  s.encode_tiled = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  s.d_err = d_err;
  s.d_sched = d_sched;
  s.sched_next = 0;
  s.capture_next = 0;
  s.ws_ok[0] = ws_ok[0];
  s.ws_ok[1] = ws_ok[1];
  s.ws_ok[2] = ws_ok[2];
  s.device = device;
  s.sm_count = prop.multiProcessorCount;
  s.inited = true;
  return ATTN_OK;
}

// attn_fwd and attn_fwd_gqa: q, out [B, T, H, D]; k, v [B, T, Hkv, D]; lse [B, H, T].
static int fwd_impl(const void* q, const void* k, const void* v, void* out, float* lse, int B, int H, int Hkv, int T,
             int D, int window, int causal, float rope_base, float eps, void* stream, const void* ve = nullptr,
             const void* x_gate = nullptr, int x_stride = 0, const void* w_gate = nullptr, float* gate_ws = nullptr,
             size_t gate_ws_bytes = 0) {
  // ---- argument checks (host only, nothing launched) ----
  if (!q || !k || !v || !out) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out)) return ATTN_ERR_INVALID_ARG;
  if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)) return ATTN_ERR_INVALID_ARG;
  if (B < 1 || H < 1 || T < 1 || D < 1) return ATTN_ERR_INVALID_ARG;
  if (Hkv < 1 || Hkv > H || H % Hkv != 0) return ATTN_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return ATTN_ERR_INVALID_ARG;
  if (!std::isfinite(rope_base) || rope_base < 0.f) return ATTN_ERR_INVALID_ARG;
  if (std::isnan(eps) || std::isinf(eps)) return ATTN_ERR_INVALID_ARG;
  const long long n_elem = static_cast<long long>(B) * T * H * D;
  if (n_elem >= (1LL << 31)) return ATTN_ERR_INVALID_ARG;
  const size_t tensor_bytes = static_cast<size_t>(n_elem) * 2;
  const size_t kv_bytes = tensor_bytes / static_cast<size_t>(H / Hkv);
  const size_t lse_bytes = static_cast<size_t>(B) * H * T * 4;
  if (overlaps(out, tensor_bytes, q, tensor_bytes) || overlaps(out, tensor_bytes, k, kv_bytes) ||
      overlaps(out, tensor_bytes, v, kv_bytes))
    return ATTN_ERR_INVALID_ARG;
  if (lse && (overlaps(lse, lse_bytes, q, tensor_bytes) || overlaps(lse, lse_bytes, k, kv_bytes) ||
              overlaps(lse, lse_bytes, v, kv_bytes) || overlaps(lse, lse_bytes, out, tensor_bytes)))
    return ATTN_ERR_INVALID_ARG;
  if (D != 32 && D != 64 && D != 128) return ATTN_ERR_UNSUPPORTED;
  if (ve) {
    if (!x_gate || !w_gate || !aligned16(ve) || !aligned16(x_gate) || !aligned16(w_gate)) return ATTN_ERR_INVALID_ARG;
    if (x_stride < 32 || x_stride % 8 != 0) return ATTN_ERR_INVALID_ARG;
    if (overlaps(out, tensor_bytes, ve, kv_bytes)) return ATTN_ERR_INVALID_ARG;
    const size_t gate_bytes = static_cast<size_t>(B) * T * Hkv * 4;
    if (!gate_ws || (reinterpret_cast<uintptr_t>(gate_ws) & 15u) || gate_ws_bytes < gate_bytes)
      return ATTN_ERR_INVALID_ARG;
    if (overlaps(gate_ws, gate_bytes, out, tensor_bytes) || (lse && overlaps(gate_ws, gate_bytes, lse, lse_bytes)))
      return ATTN_ERR_INVALID_ARG;
    if (lse && overlaps(lse, lse_bytes, ve, kv_bytes)) return ATTN_ERR_INVALID_ARG;
  }

  State& s = state();
  // Held until the launch is enqueued: the ticket slot is chosen, ordered after its previous user
  // and marked with this launch as one step, so no other thread can take the same slot in between.
  std::lock_guard<std::mutex> lock(s.mu);
  if (!s.inited) return ATTN_ERR_NOT_INITIALIZED;
  const bool use_ws = (D == 32 && s.ws_ok[0]) || (D == 64 && s.ws_ok[1]) || (D == 128 && s.ws_ok[2]);
  if (ve && !use_ws) return ATTN_ERR_UNSUPPORTED;  // the gate lives in the persistent kernel's prologue
  const float4* table = nullptr;
  int table_T = 0;
  if (rope_base > 0.f && swa_host::rope_table_locked(D, rope_base, T, &table, &table_T) != ATTN_OK) return ATTN_ERR_CUDA;

  swa::AttnParams p{};  // every field set below or zero
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.k = static_cast<const __nv_bfloat16*>(k);
  p.v = static_cast<const __nv_bfloat16*>(v);
  p.out = static_cast<__nv_bfloat16*>(out);
  p.lse = lse;
  p.rope = table;
  p.rope_T = table_T;
  p.err = s.d_err;
  p.B = B;
  p.H = H;
  p.Hkv = Hkv;
  p.kv_group = H / Hkv;
  p.T = T;
  p.window = window < 0 ? -1 : window;
  p.causal = causal;
  p.use_norm = eps >= 0.f ? 1 : 0;
  p.eps = eps >= 0.f ? eps : 0.f;
  p.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(D)));
  // With the QK-norm on, |q^|, |k^| <= sqrt(D) (after the bf16 rounding at most 2^-8 more each), so
  // every scaled score lies within sqrt(D) log2(e) (1 + 2^-8)^2; 1 % above that is the fixed softmax
  // reference of the persistent kernel.
  p.ref_log2 = eps >= 0.f ? static_cast<float>(std::sqrt(static_cast<double>(D)) * 1.4426950408889634 * 1.01) : 0.f;
  p.n_qtiles = (T + swa::kTile - 1) / swa::kTile;
  if (static_cast<long long>(B) * H * p.n_qtiles >= (1LL << 31)) return ATTN_ERR_INVALID_ARG;
  p.ve = static_cast<const __nv_bfloat16*>(ve);
  p.xg = static_cast<const __nv_bfloat16*>(x_gate);
  p.wg = static_cast<const __nv_bfloat16*>(w_gate);
  p.xg_stride = x_stride;
  p.gate = gate_ws;

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (ve) {
    // the gate factors of every (b, t, K/V head), once, before the attention kernel reads them
    const long long rows = static_cast<long long>(B) * T;
    const long long blocks = (rows + 255) / 256;
    const int grid = static_cast<int>(blocks < 8LL * s.sm_count ? blocks : 8LL * s.sm_count);
    swa::ve_gate_kernel<<<grid, 256, 0, st>>>(p);
    if (cudaGetLastError() != cudaSuccess) return ATTN_ERR_CUDA;
  }
  if (use_ws) {
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(st, &cap) != cudaSuccess) {
      cudaGetLastError();
      return ATTN_ERR_CUDA;
    }
    const bool capturing = cap != cudaStreamCaptureStatusNone;
    constexpr int kHalf = kSchedSlots / 2;
    const int idx = capturing ? kHalf + static_cast<int>(s.capture_next % kHalf)
                              : static_cast<int>(s.sched_next % kHalf);
    SchedSlot& slot = s.slots[idx];
    int* sched = s.d_sched + static_cast<size_t>(idx) * kSchedStride;
    // an eager slot last used on another stream: this launch waits for that kernel to finish first
    if (!capturing && slot.used && slot.stream != st && cudaStreamWaitEvent(st, slot.done, 0) != cudaSuccess) {
      cudaGetLastError();
      return ATTN_ERR_CUDA;
    }
    int rc;
    switch (D) {
      case 32: rc = launch_ws<32>(p, s.maps, s.encode_tiled, s.sm_count, sched, st); break;
      case 64: rc = launch_ws<64>(p, s.maps, s.encode_tiled, s.sm_count, sched, st); break;
      default: rc = launch_ws<128>(p, s.maps, s.encode_tiled, s.sm_count, sched, st); break;
    }
    if (rc != ATTN_OK) return rc;
    if (capturing) {
      ++s.capture_next;
      return ATTN_OK;
    }
    if (cudaEventRecord(slot.done, st) != cudaSuccess) {
      cudaGetLastError();
      return ATTN_ERR_CUDA;
    }
    slot.used = true;
    slot.stream = st;
    ++s.sched_next;
    return ATTN_OK;
  }
  cudaError_t e;
  switch (D) {
    case 32: e = launch_simple<32>(p, st); break;
    case 64: e = launch_simple<64>(p, st); break;
    default: e = launch_simple<128>(p, st); break;
  }
  return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

int attn_fwd(const void* q, const void* k, const void* v, void* out, float* lse, int B, int H, int T, int D,
             int window, int causal, float rope_base, float eps, void* stream) {
  return fwd_impl(q, k, v, out, lse, B, H, H, T, D, window, causal, rope_base, eps, stream);
}

int attn_fwd_gqa(const void* q, const void* k, const void* v, void* out, float* lse, int B, int H, int H_kv,
                 int T, int D, int window, int causal, float rope_base, float eps, void* stream) {
  return fwd_impl(q, k, v, out, lse, B, H, H_kv, T, D, window, causal, rope_base, eps, stream);
}

size_t attn_fwd_ve_workspace_bytes(int B, int H_kv, int T) {
  if (B < 1 || H_kv < 1 || T < 1) return 0;
  return (static_cast<size_t>(B) * T * H_kv * 4 + 255) / 256 * 256;
}

int attn_fwd_ve(const void* q, const void* k, const void* v, const void* ve, const void* x_gate, int x_stride,
                const void* w_gate, void* out, float* lse, void* workspace, size_t workspace_bytes, int B, int H,
                int H_kv, int T, int D, int window, int causal, float rope_base, float eps, void* stream) {
  if (!ve) return ATTN_ERR_INVALID_ARG;
  return fwd_impl(q, k, v, out, lse, B, H, H_kv, T, D, window, causal, rope_base, eps, stream, ve, x_gate, x_stride,
                  w_gate, static_cast<float*>(workspace), workspace_bytes);
}

int attn_fwd_kernel(int D) {
  State& s = state();
  std::lock_guard<std::mutex> lock(s.mu);
  if (!s.inited) return ATTN_ERR_NOT_INITIALIZED;
  if (D == 32) return s.ws_ok[0] ? 1 : 0;
  if (D == 64) return s.ws_ok[1] ? 1 : 0;
  if (D == 128) return s.ws_ok[2] ? 1 : 0;
  return ATTN_ERR_UNSUPPORTED;
}

void attn_destroy(void) {
  State& s = state();
  std::lock_guard<std::mutex> lock(s.mu);
  if (!s.inited) return;
  with_device(s.device, [&]() -> cudaError_t {
    for (auto& kv : s.tables)
      if (kv.second.ptr) cudaFree(kv.second.ptr);
    for (float4* ptr : s.retired) cudaFree(ptr);
    if (s.d_err) cudaFree(s.d_err);
    if (s.d_sched) cudaFree(s.d_sched);
    for (SchedSlot& sl : s.slots)
      if (sl.done) cudaEventDestroy(sl.done);
    return cudaSuccess;
  });
  for (SchedSlot& sl : s.slots) sl = SchedSlot{};
  s.maps.clear();
  s.capture_next = 0;
  s.d_sched = nullptr;
  s.ws_ok[0] = s.ws_ok[1] = s.ws_ok[2] = false;
  s.tables.clear();
  s.retired.clear();
  s.d_err = nullptr;
  s.encode_tiled = nullptr;
  s.inited = false;
  s.device = -1;
}

const char* attn_status_string(int status) {
  switch (status) {
    case ATTN_OK: return "ATTN_OK";
    case ATTN_ERR_NOT_INITIALIZED: return "ATTN_ERR_NOT_INITIALIZED";
    case ATTN_ERR_INVALID_ARG: return "ATTN_ERR_INVALID_ARG";
    case ATTN_ERR_UNSUPPORTED: return "ATTN_ERR_UNSUPPORTED";
    case ATTN_ERR_CUDA: return "ATTN_ERR_CUDA";
    case ATTN_ERR_DEVICE_TIMEOUT: return "ATTN_ERR_DEVICE_TIMEOUT";
    case ATTN_ERR_NO_DEVICE: return "ATTN_ERR_NO_DEVICE";
    case ATTN_ERR_SCRATCH_LIMIT: return "ATTN_ERR_SCRATCH_LIMIT";
    default: return "ATTN_ERR_UNKNOWN";
  }
}

int attn_selftest_wait_timeout(void* stream) {
  State& s = state();
  int* d_err = nullptr;
  int dev = -1;
  {
    std::lock_guard<std::mutex> lock(s.mu);
    if (!s.inited) return ATTN_ERR_NOT_INITIALIZED;
    d_err = s.d_err;
    dev = s.device;
  }
  cudaError_t e = with_device(dev, [&]() -> cudaError_t {
    selftest_wait_timeout_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(d_err);
    return cudaGetLastError();
  });
  return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

int attn_device_status(void) {
  State& s = state();
  std::lock_guard<std::mutex> lock(s.mu);
  if (!s.inited) return ATTN_ERR_NOT_INITIALIZED;
  int h = 0;
  cudaError_t e = with_device(s.device, [&]() -> cudaError_t {
    cudaError_t r;
    if ((r = cudaDeviceSynchronize()) != cudaSuccess) return r;
    if ((r = cudaMemcpy(&h, s.d_err, sizeof(int), cudaMemcpyDeviceToHost)) != cudaSuccess) return r;
    return cudaMemset(s.d_err, 0, sizeof(int));
  });
  if (e != cudaSuccess) return ATTN_ERR_CUDA;
  return h == 0 ? ATTN_OK : ATTN_ERR_DEVICE_TIMEOUT;
}

int attn_fwd_noalloc(const void* q, const void* k, const void* v, void* out, float* lse, int B, int H, int T,
                     int D, int window, int causal, float rope_base, float eps, void* stream) {
  // ---- the same host-side checks as attn_fwd ----
  if (!q || !k || !v || !out) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out)) return ATTN_ERR_INVALID_ARG;
  if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)) return ATTN_ERR_INVALID_ARG;
  if (B < 1 || H < 1 || T < 1 || D < 1) return ATTN_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return ATTN_ERR_INVALID_ARG;
  if (!std::isfinite(rope_base) || rope_base < 0.f) return ATTN_ERR_INVALID_ARG;
  if (std::isnan(eps) || std::isinf(eps)) return ATTN_ERR_INVALID_ARG;
  const long long n_elem = static_cast<long long>(B) * T * H * D;
  if (n_elem >= (1LL << 31)) return ATTN_ERR_INVALID_ARG;
  const size_t tensor_bytes = static_cast<size_t>(n_elem) * 2;
  const size_t lse_bytes = static_cast<size_t>(B) * H * T * 4;
  if (overlaps(out, tensor_bytes, q, tensor_bytes) || overlaps(out, tensor_bytes, k, tensor_bytes) ||
      overlaps(out, tensor_bytes, v, tensor_bytes))
    return ATTN_ERR_INVALID_ARG;
  if (lse && (overlaps(lse, lse_bytes, q, tensor_bytes) || overlaps(lse, lse_bytes, k, tensor_bytes) ||
              overlaps(lse, lse_bytes, v, tensor_bytes) || overlaps(lse, lse_bytes, out, tensor_bytes)))
    return ATTN_ERR_INVALID_ARG;
  if (D != 32 && D != 64 && D != 128) return ATTN_ERR_UNSUPPORTED;
  // ---- the fixed-size scratch bounds the cos / sin table ----
  if (rope_base > 0.f && static_cast<size_t>(T) * (D / 2) > kNoAllocTablePairs) return ATTN_ERR_SCRATCH_LIMIT;
  const int n_qtiles = (T + swa::kTile - 1) / swa::kTile;
  if (static_cast<long long>(B) * H * n_qtiles >= (1LL << 31)) return ATTN_ERR_INVALID_ARG;

  int dev = -1;
  unsigned char* scratch = nullptr;
  const int rc = noalloc_setup(&dev, &scratch);
  if (rc != ATTN_OK) return rc;

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t pairs = rope_base > 0.f ? static_cast<size_t>(T) * (D / 2) : 0;
  const int prep_blocks = static_cast<int>(pairs == 0 ? 1 : (pairs + 255) / 256 < 1184 ? (pairs + 255) / 256 : 1184);
  if (pairs > 0) {
    noalloc_prepare_kernel<<<prep_blocks, 256, 0, st>>>(scratch, T, D, rope_base);
    if (cudaGetLastError() != cudaSuccess) return ATTN_ERR_CUDA;
  }

  swa::AttnParams p{};  // every field set below or zero
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.k = static_cast<const __nv_bfloat16*>(k);
  p.v = static_cast<const __nv_bfloat16*>(v);
  p.out = static_cast<__nv_bfloat16*>(out);
  p.lse = lse;
  p.rope = rope_base > 0.f ? reinterpret_cast<const float4*>(scratch + kNoAllocHeaderBytes) : nullptr;
  p.rope_T = T;
  p.err = reinterpret_cast<int*>(scratch);
  p.B = B;
  p.H = H;
  p.Hkv = H;
  p.kv_group = 1;
  p.T = T;
  p.window = window < 0 ? -1 : window;
  p.causal = causal;
  p.use_norm = eps >= 0.f ? 1 : 0;
  p.eps = eps >= 0.f ? eps : 0.f;
  p.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(D)));
  p.n_qtiles = n_qtiles;
  cudaError_t e;
  switch (D) {
    case 32: e = launch_simple<32>(p, st); break;
    case 64: e = launch_simple<64>(p, st); break;
    default: e = launch_simple<128>(p, st); break;
  }
  return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

int attn_noalloc_status(void* stream) {
  int dev = -1;
  unsigned char* scratch = nullptr;
  const int rc = noalloc_setup(&dev, &scratch);
  if (rc != ATTN_OK) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int h = 0;
  const int zero = 0;
  // the word sits at offset 0 of the scratch array; copies to and from pageable host variables,
  // completed before returning (nothing is allocated)
  if (cudaMemcpyFromSymbolAsync(&h, g_noalloc_scratch, sizeof(int), 0, cudaMemcpyDeviceToHost, st) != cudaSuccess ||
      cudaStreamSynchronize(st) != cudaSuccess ||
      cudaMemcpyToSymbolAsync(g_noalloc_scratch, &zero, sizeof(int), 0, cudaMemcpyHostToDevice, st) != cudaSuccess ||
      cudaStreamSynchronize(st) != cudaSuccess) {
    cudaGetLastError();
    return ATTN_ERR_CUDA;
  }
  return h == 0 ? ATTN_OK : ATTN_ERR_DEVICE_TIMEOUT;
}

int attn_noalloc_selftest_wait_timeout(void* stream) {
  int dev = -1;
  unsigned char* scratch = nullptr;
  const int rc = noalloc_setup(&dev, &scratch);
  if (rc != ATTN_OK) return rc;
  selftest_wait_timeout_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(reinterpret_cast<int*>(scratch));
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

}  // extern "C"
