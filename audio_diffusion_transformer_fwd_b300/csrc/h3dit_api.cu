// C ABI of libh3dit.so: argument checks, workspace layout, tensor maps,
// kernel launches and the block / step sequencing.  The whole library is
// this one translation unit (the kernel files are included below).
#include <cuda.h>
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>

#include <algorithm>
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "../../include/h3dit.h"
#include "attention.cuh"
#include "final.cuh"
#include "gemm.cuh"
#include "gemm_i8.cuh"
#include "ptx.cuh"
#include "rows.cuh"

namespace {

using bf16 = __nv_bfloat16;

thread_local std::string t_last_error;

h3dit_status fail(h3dit_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  t_last_error = buf;
  return st;
}

// A failed runtime call is reported and then cleared from the runtime's
// last-error slot, so that it does not resurface at the next call's check.
#define H3_CUDA(call)                                                                 \
  do {                                                                                \
    cudaError_t e_ = (call);                                                          \
    if (e_ != cudaSuccess) {                                                          \
      cudaGetLastError();                                                             \
      return fail(H3DIT_E_CUDA, "%s: %s (%s:%d)", #call, cudaGetErrorString(e_),     \
                  __FILE__, __LINE__);                                                \
    }                                                                                 \
  } while (0)

#define H3_TRY(...)                        \
  do {                                     \
    h3dit_status s_ = (__VA_ARGS__);       \
    if (s_ != H3DIT_OK) return s_;         \
  } while (0)

// ------------------------------------------------------------------ fault injection
// H3DIT_FAULT=alloc|launch|arg|shape makes the block and step entry points
// fail on purpose, on the host, at the point where that failure would
// arise: alloc = the workspace is too small (E_NOMEM), arg = an argument is
// invalid (E_INVAL), shape = the shape is unsupported (E_UNSUPPORTED),
// launch = the first kernel launch fails (E_CUDA, nothing enqueued).  It
// exists to test how callers see errors; no GPU is made to fault.
enum FaultKind { kFaultNone = 0, kFaultAlloc, kFaultLaunch, kFaultArg, kFaultShape };

FaultKind injected_fault() {
  const char* e = getenv("H3DIT_FAULT");
  if (!e || !e[0]) return kFaultNone;
  if (!strcmp(e, "alloc")) return kFaultAlloc;
  if (!strcmp(e, "launch")) return kFaultLaunch;
  if (!strcmp(e, "arg")) return kFaultArg;
  if (!strcmp(e, "shape")) return kFaultShape;
  return kFaultNone;
}

// The next BF16 GEMM launch (any thread) gets this k-block as its stall
// point (h3dit_test_stall_next_gemm); -1 = none.
std::atomic<int> g_stall_request{-1};
int take_stall_request() { return g_stall_request.exchange(-1); }

// ------------------------------------------------------------------ tracing
// NVTX ranges around every block and step (free unless a profiler that
// records NVTX is attached): "h3dit block b" nests inside "h3dit step".
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  NvtxRange(const char* prefix, int index) {
    char buf[48];
    snprintf(buf, sizeof(buf), "%s %d", prefix, index);
    nvtxRangePushA(buf);
  }
  ~NvtxRange() { nvtxRangePop(); }
};

// ------------------------------------------------------------------ timing
enum KernelClass { kRows = 0, kQKV = 1, kAttn = 2, kOProj = 3, kFC1 = 4, kFC2 = 5, kReduce = 6, kQuant = 7, kNumClasses = 8 };

struct Timing {
  std::mutex mu;
  bool enabled = false;
  struct Pending { int cls; cudaEvent_t a, b; int kernels; };
  std::vector<Pending> pending;
  double total_ms[kNumClasses] = {0};
  long long count[kNumClasses] = {0};
} g_timing;

struct TimedLaunch {
  int cls;
  cudaStream_t s;
  cudaEvent_t a = nullptr, b = nullptr;
  int kernels = 1;   // kernel launches between the two events
  TimedLaunch(int c, cudaStream_t st) : cls(c), s(st) {
    if (!g_timing.enabled) return;
    cudaEventCreate(&a);
    cudaEventCreate(&b);
    cudaEventRecord(a, s);
  }
  ~TimedLaunch() {
    if (!a) return;
    cudaEventRecord(b, s);
    std::lock_guard<std::mutex> lk(g_timing.mu);
    g_timing.pending.push_back({cls, a, b, kernels});
  }
};

// ------------------------------------------------------------------ device facts
int sm_count() {
  static int cached[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return 148;
  if (cached[dev] == 0) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    cached[dev] = n > 0 ? n : 148;
  }
  return cached[dev];
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

h3dit_status get_encoder(EncodeTiledFn* out) {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  static cudaError_t err = cudaSuccess;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    err = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q);
    if (err == cudaSuccess && q == cudaDriverEntryPointSuccess) fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  if (!fn) return fail(H3DIT_E_CUDA, "cuTensorMapEncodeTiled unavailable (%s)", cudaGetErrorString(err));
  *out = fn;
  return H3DIT_OK;
}

// BF16 tensor map with the 128-byte swizzle; dims/strides innermost first,
// strides in bytes for dims 1.. ; out-of-bounds boxes read zeros.
h3dit_status make_map(CUtensorMap* m, const void* base, int rank, const uint64_t* dims,
                      const uint64_t* strides, const uint32_t* box) {
  EncodeTiledFn enc;
  H3_TRY(get_encoder(&enc));
  cuuint64_t gd[3], gs[2];
  cuuint32_t bx[3], es[3] = {1, 1, 1};
  for (int i = 0; i < rank; ++i) { gd[i] = dims[i]; bx[i] = box[i]; }
  for (int i = 0; i < rank - 1; ++i) gs[i] = strides[i];
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(base), gd, gs, bx, es,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(H3DIT_E_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  return H3DIT_OK;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Which projections run on int8 codes ([linlog] "int8 量化": the MLP alone,
// QKV alone, or all four).
struct Int8Set {
  bool qkv = false, o = false, fc1 = false, fc2 = false;
  bool any() const { return qkv || o || fc1 || fc2; }
};
Int8Set int8_set(int precision) {
  Int8Set q;
  switch (precision) {
    case H3DIT_INT8: q.qkv = q.o = q.fc1 = q.fc2 = true; break;
    case H3DIT_INT8_MLP: q.fc1 = q.fc2 = true; break;
    case H3DIT_INT8_QKV: q.qkv = true; break;
    default: break;
  }
  return q;
}

// ------------------------------------------------------------------ config checks
h3dit_status check_cfg(const h3dit_config* c) {
  if (!c) return fail(H3DIT_E_INVAL, "config is NULL");
  if (c->d <= 0 || c->heads <= 0 || c->head_dim <= 0 || c->ffn <= 0)
    return fail(H3DIT_E_INVAL, "non-positive block size");
  if (c->heads * c->head_dim != c->d) return fail(H3DIT_E_INVAL, "heads*head_dim != d");
  if (c->head_dim != 64 && c->head_dim != 128)
    return fail(H3DIT_E_UNSUPPORTED, "head_dim %d (64 or 128 supported)", c->head_dim);
  if (c->d % 256 != 0 || c->d > 8192) return fail(H3DIT_E_UNSUPPORTED, "d %d (multiple of 256, <= 8192)", c->d);
  if (c->ffn % 256 != 0) return fail(H3DIT_E_UNSUPPORTED, "ffn %d (multiple of 256)", c->ffn);
  int s = 0;
  for (int i = 0; i < 3; ++i) {
    if (c->rope_sections[i] < 0 || c->rope_sections[i] % 2 != 0)
      return fail(H3DIT_E_INVAL, "rope section %d must be even and >= 0", i);
    s += c->rope_sections[i];
  }
  if (s != c->head_dim) return fail(H3DIT_E_INVAL, "rope sections sum %d != head_dim %d", s, c->head_dim);
  if (!(c->eps > 0.f)) return fail(H3DIT_E_INVAL, "eps must be > 0");
  if (!(c->rope_theta > 0.f)) return fail(H3DIT_E_INVAL, "rope_theta must be > 0");
  if (c->precision < H3DIT_BF16 || c->precision > H3DIT_INT8_QKV)
    return fail(H3DIT_E_INVAL, "precision %d", c->precision);
  if (int8_set(c->precision).fc2 && c->ffn > 1024 && c->ffn % 1024 != 0)
    return fail(H3DIT_E_UNSUPPORTED, "int8 ffn %d (FC2 scale groups of 1024 need ffn <= 1024 or a multiple of 1024)",
                c->ffn);
  return H3DIT_OK;
}

// Attention alone needs only the head layout.
h3dit_status check_heads(const h3dit_config* c) {
  if (!c) return fail(H3DIT_E_INVAL, "config is NULL");
  if (c->heads <= 0 || c->head_dim <= 0) return fail(H3DIT_E_INVAL, "non-positive head layout");
  if (c->head_dim != 64 && c->head_dim != 128)
    return fail(H3DIT_E_UNSUPPORTED, "head_dim %d (64 or 128 supported)", c->head_dim);
  if (c->d != c->heads * c->head_dim) return fail(H3DIT_E_INVAL, "heads*head_dim != d");
  return H3DIT_OK;
}

h3dit_status check_grid(const h3dit_video_grid* g, int n_tokens) {
  if (!g) return fail(H3DIT_E_INVAL, "video grid is NULL");
  if (g->offset < 0 || g->T < 0 || g->Hh < 0 || g->W < 0)
    return fail(H3DIT_E_INVAL, "negative video grid field");
  const long long nv = 1LL * g->T * g->Hh * g->W;
  if (g->offset + nv > n_tokens) return fail(H3DIT_E_INVAL, "video grid exceeds the %d rows", n_tokens);
  return H3DIT_OK;
}

h3::PairGrid pair_grid(const h3dit_video_grid* g, int n_tokens) {
  h3::PairGrid p;
  p.offset = g->offset;
  p.T = g->T;
  p.Hh = g->Hh;
  p.W = g->W;
  p.Wr = (g->W + 1) / 2;
  p.n_full = n_tokens;
  p.n_red = n_tokens - g->T * g->Hh * (g->W - p.Wr);
  return p;
}

// ------------------------------------------------------------------ launches
template <typename K>
h3dit_status set_smem(K kernel, size_t bytes) {
  // Dynamic shared memory above 48 KB is opted into per kernel and per
  // device: once per (kernel, device) pair, whatever thread gets there first.
  static std::mutex mu;
  static std::vector<std::pair<const void*, uint64_t>> done;   // kernel -> bit per device ordinal
  int dev = 0;
  H3_CUDA(cudaGetDevice(&dev));
  if (dev < 0 || dev >= 64) return fail(H3DIT_E_UNSUPPORTED, "device ordinal %d out of range", dev);
  const void* key = reinterpret_cast<const void*>(kernel);
  std::lock_guard<std::mutex> lk(mu);
  auto it = std::find_if(done.begin(), done.end(), [&](const std::pair<const void*, uint64_t>& e) {
    return e.first == key;
  });
  if (it != done.end() && (it->second >> dev & 1u)) return H3DIT_OK;
  H3_CUDA(cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes));
  if (it == done.end()) done.emplace_back(key, 0);
  for (auto& e : done)
    if (e.first == key) e.second |= uint64_t(1) << dev;
  return H3DIT_OK;
}

// Tensor maps of the GEMM operands A [M][K] and B [N][K] (BF16, K-major) and
// the tile counts; shared by the BF16 and the int8-code kernels.
// Width of the projections' tile raster in N-tiles: 16 unless H3DIT_GEMM_BAND
// names another width (1..64; a tuning switch, read at every launch).
int gemm_band() {
  const char* e = getenv("H3DIT_GEMM_BAND");
  const int v = e ? atoi(e) : 0;
  return (v >= 1 && v <= 64) ? v : h3::kGemmGroupN;
}

h3dit_status gemm_setup(const void* A, const void* B, int M, int N, int K, CUtensorMap& ta, CUtensorMap& tb,
                        h3::GemmArgs& args) {
  if (M < 1 || N % h3::kGemmBN != 0 || K % h3::kGemmBK != 0 || N <= 0 || K <= 0)
    return fail(H3DIT_E_UNSUPPORTED, "gemm shape %dx%dx%d (n %% 256, k %% 64)", M, N, K);
  if (!aligned(A, 16) || !aligned(B, 16)) return fail(H3DIT_E_INVAL, "gemm operands must be 16-byte aligned");
  {
    const uint64_t dims[2] = {(uint64_t)K, (uint64_t)M};
    const uint64_t str[1] = {(uint64_t)K * 2};
    const uint32_t box[2] = {h3::kGemmBK, h3::kGemmBM};
    H3_TRY(make_map(&ta, A, 2, dims, str, box));
  }
  {
    const uint64_t dims[2] = {(uint64_t)K, (uint64_t)N};
    const uint64_t str[1] = {(uint64_t)K * 2};
    const uint32_t box[2] = {h3::kGemmBK, h3::kGemmBN};
    H3_TRY(make_map(&tb, B, 2, dims, str, box));
  }
  args.M = M;
  args.N = N;
  args.K = K;
  args.stall_kb = -1;
  args.band_n = gemm_band();
  args.tiles_m = (M + h3::kGemmBM - 1) / h3::kGemmBM;
  args.tiles_n = N / h3::kGemmBN;
  args.num_tiles = args.tiles_m * args.tiles_n;
  args.full_tiles = args.num_tiles;
  args.num_units = args.num_tiles;
  return H3DIT_OK;
}

// Which BF16 projection kernel runs: the CTA-pair kernel unless
// H3DIT_GEMM_SINGLE_CTA=1 selects the single-CTA one (an A/B switch, read at
// every launch; both kernels give the same bits).
bool gemm_pair_enabled() {
  const char* e = getenv("H3DIT_GEMM_SINGLE_CTA");
  return !(e && e[0] && e[0] != '0');
}

// Clusters of two CTA-pair GEMM CTAs that fit the device at once (the
// persistent grid's size), per kernel and device.
template <typename K>
h3dit_status pair_clusters(K kernel, int threads, size_t smem_bytes, int* out) {
  static std::mutex mu;
  static std::vector<std::pair<std::pair<const void*, int>, int>> cache;
  int dev = 0;
  H3_CUDA(cudaGetDevice(&dev));
  const void* key = reinterpret_cast<const void*>(kernel);
  std::lock_guard<std::mutex> lk(mu);
  for (auto& e : cache)
    if (e.first.first == key && e.first.second == dev) {
      *out = e.second;
      return H3DIT_OK;
    }
  cudaLaunchConfig_t lc{};
  lc.gridDim = dim3(2 * (sm_count() / 2));
  lc.blockDim = dim3(threads);
  lc.dynamicSmemBytes = smem_bytes;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  lc.attrs = attr;
  lc.numAttrs = 1;
  int n = 0;
  H3_CUDA(cudaOccupancyMaxActiveClusters(&n, kernel, &lc));
  if (n < 1) return fail(H3DIT_E_CUDA, "no CTA pair of the projection kernel fits the device");
  cache.push_back({{key, dev}, n});
  *out = n;
  return H3DIT_OK;
}

// Kernels of the block and the step are launched with programmatic stream
// serialisation: each may be scheduled as the one before it retires its
// CTAs, runs its prologue (barriers, tensor memory, tensor-map prefetch)
// and waits in grid_dep_wait() for that kernel before touching global
// memory (measured 0.4 % off the block).  H3DIT_PDL=0 launches them in plain
// stream order (an A/B switch read at every launch).  Only kernels that call
// grid_dep_wait() first go through launch_ex.
bool pdl_enabled() {
  const char* e = getenv("H3DIT_PDL");
  return !(e && e[0] == '0');
}

template <typename K, typename... A>
h3dit_status launch_ex(K kernel, dim3 grid, dim3 block, size_t smem_bytes, cudaStream_t s, int cluster_x,
                       A... args) {
  cudaLaunchConfig_t lc{};
  lc.gridDim = grid;
  lc.blockDim = block;
  lc.dynamicSmemBytes = smem_bytes;
  lc.stream = s;
  cudaLaunchAttribute attr[2];
  int na = 0;
  if (cluster_x > 1) {
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = cluster_x;
    attr[na].val.clusterDim.y = 1;
    attr[na].val.clusterDim.z = 1;
    ++na;
  }
  if (pdl_enabled()) {
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  lc.attrs = attr;
  lc.numAttrs = na;
  H3_CUDA(cudaLaunchKernelEx(&lc, kernel, args...));
  return H3DIT_OK;
}

// A persistent kernel on CTA pairs: as many clusters of two as fit the
// device at once (at most one per tile), each walking tiles cluster,
// cluster + clusters, ...
template <typename K, typename... A>
h3dit_status launch_on_pairs(K kernel, int threads, size_t smem_bytes, int tiles, cudaStream_t s, A... args) {
  H3_TRY(set_smem(kernel, smem_bytes));
  int fit = 0;
  H3_TRY(pair_clusters(kernel, threads, smem_bytes, &fit));
  const int clusters = std::min(tiles, fit);
  return launch_ex(kernel, dim3(2 * clusters), dim3(threads), smem_bytes, s, 2, args...);
}

// The last wave of whole tiles split into 256 x 128 halves when it would
// leave at least half of the pairs idle (default; H3DIT_GEMM_TAIL=0 keeps
// whole tiles, an A/B switch read at every launch).
bool gemm_tail_split() {
  const char* e = getenv("H3DIT_GEMM_TAIL");
  return !(e && e[0] == '0');
}

// On `fit` co-resident pairs: the last wave of whole tiles becomes half
// tiles when it would keep at most half of the pairs busy.
void split_tail(h3::GemmArgs& args, int fit) {
  const int rem = args.num_tiles % fit;
  args.full_tiles = args.num_tiles;
  if (gemm_tail_split() && args.num_tiles > fit && rem > 0 && 2 * rem <= fit) args.full_tiles = args.num_tiles - rem;
  args.num_units = args.full_tiles + 2 * (args.num_tiles - args.full_tiles);
}

template <int EPI>
h3dit_status launch_pair_kernel(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tbh,
                                h3::GemmArgs args, cudaStream_t s) {
  auto kernel = h3::gemm_bf16_pair_kernel<EPI>;
  H3_TRY(set_smem(kernel, h3::kPairSmemBytes));
  int fit = 0;
  H3_TRY(pair_clusters(kernel, h3::kGemmThreads, h3::kPairSmemBytes, &fit));
  split_tail(args, fit);
  return launch_on_pairs(kernel, h3::kGemmThreads, h3::kPairSmemBytes, args.num_units, s, ta, tb, tbh, args);
}

// Tensor maps and tile counts of a projection on CTA pairs: 256 x 256
// output tiles, each CTA of a pair loading 128 A rows and 128 of the tile's
// 256 weight rows per k-block.
h3dit_status pair_setup(const void* A, const void* B, int M, int N, int K, CUtensorMap& ta, CUtensorMap& tb,
                        h3::GemmArgs& args) {
  if (M < 1 || N % h3::kGemmBN != 0 || K % h3::kGemmBK != 0 || N <= 0 || K <= 0)
    return fail(H3DIT_E_UNSUPPORTED, "gemm shape %dx%dx%d (n %% 256, k %% 64)", M, N, K);
  if (!aligned(A, 16) || !aligned(B, 16)) return fail(H3DIT_E_INVAL, "gemm operands must be 16-byte aligned");
  {
    const uint64_t dims[2] = {(uint64_t)K, (uint64_t)M};
    const uint64_t str[1] = {(uint64_t)K * 2};
    const uint32_t box[2] = {h3::kGemmBK, h3::kPairRows};
    H3_TRY(make_map(&ta, A, 2, dims, str, box));
  }
  {
    const uint64_t dims[2] = {(uint64_t)K, (uint64_t)N};
    const uint64_t str[1] = {(uint64_t)K * 2};
    const uint32_t box[2] = {h3::kGemmBK, h3::kPairRows};
    H3_TRY(make_map(&tb, B, 2, dims, str, box));
  }
  args.M = M;
  args.N = N;
  args.K = K;
  args.stall_kb = -1;
  args.band_n = gemm_band();
  args.tiles_m = (M + 2 * h3::kPairRows - 1) / (2 * h3::kPairRows);
  args.tiles_n = N / h3::kGemmBN;
  args.num_tiles = args.tiles_m * args.tiles_n;
  args.full_tiles = args.num_tiles;
  args.num_units = args.num_tiles;
  return H3DIT_OK;
}

// Weight tiles of a half unit on CTA pairs: 64 rows per CTA.
h3dit_status half_weight_map(const void* B, int N, int K, CUtensorMap& tbh) {
  const uint64_t dims[2] = {(uint64_t)K, (uint64_t)N};
  const uint64_t str[1] = {(uint64_t)K * 2};
  const uint32_t box[2] = {h3::kGemmBK, h3::kPairRows / 2};
  return make_map(&tbh, B, 2, dims, str, box);
}

h3dit_status launch_gemm_pair(int epi, const void* A, const void* B, int M, int N, int K, h3::GemmArgs args,
                              int cls, cudaStream_t s) {
  CUtensorMap ta, tb, tbh;
  H3_TRY(pair_setup(A, B, M, N, K, ta, tb, args));
  H3_TRY(half_weight_map(B, N, K, tbh));
  args.stall_kb = take_stall_request();
  if (args.stall_kb >= K / h3::kGemmBK) args.stall_kb = -1;
  TimedLaunch tl(cls, s);
  switch (epi) {
    case h3::kEpiStore: H3_TRY(launch_pair_kernel<h3::kEpiStore>(ta, tb, tbh, args, s)); break;
    case h3::kEpiGelu: H3_TRY(launch_pair_kernel<h3::kEpiGelu>(ta, tb, tbh, args, s)); break;
    case h3::kEpiQKV: H3_TRY(launch_pair_kernel<h3::kEpiQKV>(ta, tb, tbh, args, s)); break;
    default: return fail(H3DIT_E_INVAL, "unknown epilogue %d", epi);
  }
  H3_CUDA(cudaGetLastError());
  return H3DIT_OK;
}

h3dit_status launch_gemm(int epi, const void* A, const void* B, int M, int N, int K, h3::GemmArgs args,
                         int cls, cudaStream_t s) {
  if (gemm_pair_enabled()) return launch_gemm_pair(epi, A, B, M, N, K, args, cls, s);
  CUtensorMap ta, tb;
  H3_TRY(gemm_setup(A, B, M, N, K, ta, tb, args));
  args.stall_kb = take_stall_request();
  if (args.stall_kb >= args.K / h3::kGemmBK) args.stall_kb = -1;
  const int grid = std::min(args.num_tiles, sm_count());
  TimedLaunch tl(cls, s);
  switch (epi) {
    case h3::kEpiStore: {
      H3_TRY(set_smem(h3::gemm_bf16_tc_kernel<h3::kEpiStore>, h3::kGemmSmemBytes));
      h3::gemm_bf16_tc_kernel<h3::kEpiStore><<<grid, h3::kGemmThreads, h3::kGemmSmemBytes, s>>>(ta, tb, args);
      break;
    }
    case h3::kEpiGelu: {
      H3_TRY(set_smem(h3::gemm_bf16_tc_kernel<h3::kEpiGelu>, h3::kGemmSmemBytes));
      h3::gemm_bf16_tc_kernel<h3::kEpiGelu><<<grid, h3::kGemmThreads, h3::kGemmSmemBytes, s>>>(ta, tb, args);
      break;
    }
    case h3::kEpiQKV: {
      H3_TRY(set_smem(h3::gemm_bf16_tc_kernel<h3::kEpiQKV>, h3::kGemmSmemBytes));
      h3::gemm_bf16_tc_kernel<h3::kEpiQKV><<<grid, h3::kGemmThreads, h3::kGemmSmemBytes, s>>>(ta, tb, args);
      break;
    }
    default:
      return fail(H3DIT_E_INVAL, "unknown epilogue %d", epi);
  }
  H3_CUDA(cudaGetLastError());
  return H3DIT_OK;
}

template <int EPI, int MODE>
h3dit_status launch_i8_kernel(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tbh,
                              h3::GemmArgs args, const h3::I8Args& qa, bool pair, cudaStream_t s) {
  if (pair) {
    auto kernel = h3::gemm_i8x_tc_kernel<EPI, MODE, true>;
    H3_TRY(set_smem(kernel, h3::kPairSmemBytes));
    int fit = 0;
    H3_TRY(pair_clusters(kernel, h3::kI8Threads, h3::kPairSmemBytes, &fit));
    split_tail(args, fit);
    H3_TRY(launch_on_pairs(kernel, h3::kI8Threads, h3::kPairSmemBytes, args.num_units, s, ta, tb, tbh, args, qa));
  } else {
    const int grid = std::min(args.num_tiles, sm_count());
    H3_TRY(set_smem(h3::gemm_i8x_tc_kernel<EPI, MODE, false>, h3::kGemmSmemBytes));
    h3::gemm_i8x_tc_kernel<EPI, MODE, false><<<grid, h3::kI8Threads, h3::kGemmSmemBytes, s>>>(ta, tb, tb, args,
                                                                                              qa);
  }
  H3_CUDA(cudaGetLastError());
  return H3DIT_OK;
}

// Projection on int8 codes held as BF16 values (see gemm_i8.cuh).  group ==
// K: per-row activation scales sa [M], int32 accumulation over chunks of
// 1024; group < K: sa [M][K / group], one chunk per group (group % 64 == 0,
// group <= 1024).  epi kEpiAcc writes the raw int32 accumulators.
h3dit_status launch_gemm_i8(int epi, const void* A, const float* sa, int group, const void* B, const float* sb,
                            int M, int N, int K, h3::GemmArgs args, int32_t* acc, int cls, cudaStream_t s) {
  CUtensorMap ta, tb, tbh;
  const bool pair = gemm_pair_enabled();
  if (pair) {
    H3_TRY(pair_setup(A, B, M, N, K, ta, tb, args));
    H3_TRY(half_weight_map(B, N, K, tbh));
  } else {
    H3_TRY(gemm_setup(A, B, M, N, K, ta, tb, args));
    tbh = tb;
  }
  if (K > (1 << 17)) return fail(H3DIT_E_UNSUPPORTED, "int8 k %d (the int32 accumulator bound needs k <= 131072)", K);
  h3::I8Args qa{};
  qa.sa = sa;
  qa.sb = sb;
  qa.acc = acc;
  const bool grouped = group != K;
  if (grouped) {
    if (group < 64 || group % 64 != 0 || group > 1024 || K % group != 0)
      return fail(H3DIT_E_UNSUPPORTED, "int8 group %d (a multiple of 64, <= 1024, dividing k %d)", group, K);
    if (epi == h3::kEpiAcc) return fail(H3DIT_E_INVAL, "raw accumulators are per-row-scale only");
    qa.chunk_kb = group / h3::kGemmBK;
    qa.groups = K / group;
  } else {
    qa.chunk_kb = h3::kI8MaxChunkKb;
    qa.groups = 1;
  }
  if (epi != h3::kEpiAcc && (!sa || !sb || !aligned(sb, 16)))
    return fail(H3DIT_E_INVAL, "int8 scales missing or sb not 16-byte aligned");
  TimedLaunch tl(cls, s);
  if (grouped) {
    switch (epi) {
      case h3::kEpiStore: return launch_i8_kernel<h3::kEpiStore, h3::kI8Group>(ta, tb, tbh, args, qa, pair, s);
      case h3::kEpiGelu: return launch_i8_kernel<h3::kEpiGelu, h3::kI8Group>(ta, tb, tbh, args, qa, pair, s);
      default: return fail(H3DIT_E_INVAL, "grouped int8 epilogue %d", epi);
    }
  }
  switch (epi) {
    case h3::kEpiStore: return launch_i8_kernel<h3::kEpiStore, h3::kI8Int>(ta, tb, tbh, args, qa, pair, s);
    case h3::kEpiGelu: return launch_i8_kernel<h3::kEpiGelu, h3::kI8Int>(ta, tb, tbh, args, qa, pair, s);
    case h3::kEpiQKV: return launch_i8_kernel<h3::kEpiQKV, h3::kI8Int>(ta, tb, tbh, args, qa, pair, s);
    case h3::kEpiAcc: return launch_i8_kernel<h3::kEpiAcc, h3::kI8Int>(ta, tb, tbh, args, qa, pair, s);
    default: return fail(H3DIT_E_INVAL, "int8 epilogue %d", epi);
  }
}

// The key split of a short last wave of attention units (default;
// H3DIT_ATTN_SPLIT=0 runs whole units only: an A/B switch read at every call).
bool attn_split_enabled() {
  const char* e = getenv("H3DIT_ATTN_SPLIT");
  return !(e && e[0] == '0');
}

// Attention's full waves on persistent CTAs (default; H3DIT_ATTN_PERSIST=0
// one CTA per unit, an A/B switch read at every call, same bits).
bool attn_persistent() {
  const char* e = getenv("H3DIT_ATTN_PERSIST");
  return !(e && e[0] == '0');
}

h3dit_status launch_attention(const h3dit_config* c, const void* q, const void* k, const void* vt, int vt_ld,
                              int n, void* o, cudaStream_t s) {
  const int dh = c->head_dim, H = c->heads;
  if (vt_ld < n || vt_ld % 8 != 0) return fail(H3DIT_E_INVAL, "vt_ld %d (>= n, multiple of 8)", vt_ld);
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(vt, 16) || !aligned(o, 16))
    return fail(H3DIT_E_INVAL, "attention tensors must be 16-byte aligned");
  CUtensorMap tq, tk, tv;
  {
    const uint64_t dims[3] = {(uint64_t)dh, (uint64_t)n, (uint64_t)H};
    const uint64_t str[2] = {(uint64_t)dh * 2, (uint64_t)n * dh * 2};
    const uint32_t box[3] = {64, h3::kAttnBQ, 1};
    H3_TRY(make_map(&tq, q, 3, dims, str, box));
    H3_TRY(make_map(&tk, k, 3, dims, str, box));
  }
  {
    const uint64_t dims[3] = {(uint64_t)n, (uint64_t)dh, (uint64_t)H};
    const uint64_t str[2] = {(uint64_t)vt_ld * 2, (uint64_t)dh * vt_ld * 2};
    const uint32_t box[3] = {64, (uint32_t)dh, 1};
    H3_TRY(make_map(&tv, vt, 3, dims, str, box));
  }
  h3::AttnArgs a;
  a.n = n;
  a.heads = H;
  a.o = static_cast<bf16*>(o);
  a.scale_log2 = 1.4426950408889634f / sqrtf((float)dh);
  // One CTA (one per SM: its shared memory) per unit of 256 query rows of a
  // head.  When the last wave of units would keep at most half of the SMs
  // busy, those units run as CTA pairs that split the keys in two and
  // combine their partial results, so the tail takes about half a wave.
  const int rows_per_cta = h3::kAttnTilesQ * h3::kAttnBQ;
  a.qpairs = (n + rows_per_cta - 1) / rows_per_cta;
  const long long units = 1LL * a.qpairs * H;
  if (units > 0x3fffffffLL) return fail(H3DIT_E_UNSUPPORTED, "attention: %lld units", units);
  const int nkv = (n + h3::kAttnBKV - 1) / h3::kAttnBKV;
  const int sms = sm_count();
  const int rem = static_cast<int>(units % sms);
  const int tail = (attn_split_enabled() && units > sms && rem > 0 && 2 * rem <= sms && nkv >= 2) ? rem : 0;
  const int full = static_cast<int>(units) - tail;
  TimedLaunch tl(kAttn, s);
  // The full waves run persistent: min(units, SMs) CTAs, each walking
  // units first, first + grid, ... so that a CTA loads its next unit's
  // query and first key tiles while it finishes the current one.
  auto run = [&](auto kernel, size_t smem) -> h3dit_status {
    H3_TRY(set_smem(kernel, smem));
    a.unit0 = 0;
    a.units = full;
    a.split = 0;
    if (full > 0)
      H3_TRY(launch_ex(kernel, dim3(std::min(full, attn_persistent() ? sms : full)), dim3(h3::kAttnThreads), smem,
                       s, 1, tq, tk, tv, a));
    tl.kernels = (full > 0 ? 1 : 0) + (tail > 0 ? 1 : 0);
    if (tail > 0) {
      a.unit0 = full;
      a.units = tail;
      a.split = 1;
      H3_TRY(launch_ex(kernel, dim3(2 * tail), dim3(h3::kAttnThreads), smem, s, 2, tq, tk, tv, a));
    }
    return H3DIT_OK;
  };
  if (dh == 128) H3_TRY(run(h3::attn_fwd_tc_kernel<128>, h3::AttnSmem<128>::kTotal));
  else H3_TRY(run(h3::attn_fwd_tc_kernel<64>, h3::AttnSmem<64>::kTotal));
  return H3DIT_OK;
}

bool fusion_disabled() {
  static int v = -1;
  if (v < 0) {
    const char* e = getenv("H3DIT_DISABLE_GATED_ADALN");
    v = (e && e[0] && e[0] != '0') ? 1 : 0;
  }
  return v == 1;
}

template <bool GATE, bool NORM, bool QUANT>
h3dit_status launch_row_kernel(int nv, bf16* x, const bf16* branch, const float* gate, const float* shift,
                               const float* scale, bf16* h, float* hs, int n, int d, float eps,
                               const h3::SegMap& sm, cudaStream_t s) {
#define H3_ROW_CASE(NVV)                                                                                  \
  case NVV:                                                                                               \
    return launch_ex(h3::gate_adaln_kernel<GATE, NORM, QUANT, NVV>, dim3(n), dim3(h3::kRowThreads), 0, s, 1, \
                     x, branch, gate, shift, scale, h, hs, d, eps, sm);
  switch (nv) {
    H3_ROW_CASE(1) H3_ROW_CASE(2) H3_ROW_CASE(3) H3_ROW_CASE(4)
    H3_ROW_CASE(5) H3_ROW_CASE(6) H3_ROW_CASE(7) default: H3_ROW_CASE(8)
  }
#undef H3_ROW_CASE
}

// Gated residual (branch != NULL) and/or AdaLN (shift != NULL).  hs != NULL
// selects the int8 form of the AdaLN output: h receives the row's int8 codes
// as BF16 values and hs[row] the scale.
h3::SegMap one_segment() {
  h3::SegMap m{};
  m.count = 1;
  return m;
}

h3dit_status launch_rows(void* x, const void* branch, const float* gate, const float* shift, const float* scale,
                         void* h, float* hs, int n, int d, float eps, cudaStream_t s,
                         const h3::SegMap& sm = one_segment()) {
  TimedLaunch tl(kRows, s);
  bf16* xb = static_cast<bf16*>(x);
  const bf16* bb = static_cast<const bf16*>(branch);
  bf16* hb = static_cast<bf16*>(h);
  const bool gate_on = branch != nullptr;
  const bool norm_on = shift != nullptr;
  const bool quant = hs != nullptr;
  if (d % 8 != 0 || d > h3::kRowMaxVec * h3::kRowThreads * 8)
    return fail(H3DIT_E_UNSUPPORTED, "row width %d (multiple of 8, <= 8192)", d);
  const int nv = (d / 8 + h3::kRowThreads - 1) / h3::kRowThreads;
  if (gate_on && norm_on && !fusion_disabled()) {
    if (quant)
      H3_TRY(launch_row_kernel<true, true, true>(nv, xb, bb, gate, shift, scale, hb, hs, n, d, eps, sm, s));
    else
      H3_TRY(launch_row_kernel<true, true, false>(nv, xb, bb, gate, shift, scale, hb, nullptr, n, d, eps, sm, s));
  } else {
    tl.kernels = (gate_on ? 1 : 0) + (norm_on ? 1 : 0);
    if (gate_on)
      H3_TRY(launch_row_kernel<true, false, false>(nv, xb, bb, gate, nullptr, nullptr, nullptr, nullptr, n, d, eps,
                                                   sm, s));
    if (norm_on) {
      if (quant)
        H3_TRY(launch_row_kernel<false, true, true>(nv, xb, nullptr, nullptr, shift, scale, hb, hs, n, d, eps, sm,
                                                    s));
      else
        H3_TRY(launch_row_kernel<false, true, false>(nv, xb, nullptr, nullptr, shift, scale, hb, nullptr, n, d, eps,
                                                     sm, s));
    }
  }
  H3_CUDA(cudaGetLastError());
  return H3DIT_OK;
}

// Groups of 256, 512, 768 or 1024 columns: one warp per group (quantize_warp_kernel).
template <bool CODES>
// *done = false (nothing launched) for other group sizes.
h3dit_status launch_quantize_warp(const void* x, int rows, int cols, int group, bf16* q16, int8_t* q8,
                                  float* scales, cudaStream_t s, bool* done) {
  *done = false;
  if (group % 256 != 0 || group > 1024) return H3DIT_OK;
  *done = true;
  const long long n_groups = 1LL * rows * (cols / group);
  const dim3 blocks((unsigned)((n_groups + 7) / 8));
  const bf16* xb = static_cast<const bf16*>(x);
  switch (group / 256) {
    case 1: return launch_ex(h3::quantize_warp_kernel<1, CODES>, blocks, dim3(256), 0, s, 1, xb, cols, group, n_groups,
                             q16, q8, scales);
    case 2: return launch_ex(h3::quantize_warp_kernel<2, CODES>, blocks, dim3(256), 0, s, 1, xb, cols, group, n_groups,
                             q16, q8, scales);
    case 3: return launch_ex(h3::quantize_warp_kernel<3, CODES>, blocks, dim3(256), 0, s, 1, xb, cols, group, n_groups,
                             q16, q8, scales);
    default: return launch_ex(h3::quantize_warp_kernel<4, CODES>, blocks, dim3(256), 0, s, 1, xb, cols, group,
                              n_groups, q16, q8, scales);
  }
}

h3dit_status launch_quantize_codes(const void* x, int rows, int cols, int group, void* q, float* scales,
                                   cudaStream_t s) {
  const long long blocks = 1LL * rows * (cols / group);
  if (blocks > 0x7fffffffLL) return fail(H3DIT_E_UNSUPPORTED, "too many groups");
  TimedLaunch tl(kQuant, s);
  bool done = false;
  H3_TRY(launch_quantize_warp<true>(x, rows, cols, group, static_cast<bf16*>(q), nullptr, scales, s, &done));
  if (!done)
    H3_TRY(launch_ex(h3::quantize_codes_kernel, dim3((unsigned)blocks), dim3(h3::kRowThreads), 0, s, 1,
                     static_cast<const bf16*>(x), cols, group, static_cast<bf16*>(q), scales));
  return H3DIT_OK;
}

h3dit_status launch_rope_table(const h3dit_config* c, const float* pos, int n, float* table, cudaStream_t s) {
  if (injected_fault() == kFaultLaunch) return fail(H3DIT_E_CUDA, "injected launch failure (H3DIT_FAULT=launch)");
  TimedLaunch tl(kRows, s);
  h3::RopeSpec rs;
  rs.head_dim = c->head_dim;
  for (int i = 0; i < 3; ++i) rs.sec[i] = c->rope_sections[i];
  rs.theta = c->rope_theta;
  const int total = n * (c->head_dim / 2);
  H3_TRY(launch_ex(h3::rope_table_kernel, dim3((total + 255) / 256), dim3(256), 0, s, 1, pos, n, rs,
                   reinterpret_cast<float2*>(table)));
  return H3DIT_OK;
}

// ------------------------------------------------------------------ workspace
struct Arena {
  size_t a1 = 0, a2 = 0, a3 = 0, rope = 0;     // offsets
  size_t xred = 0, rope_red = 0, pos_red = 0;  // reduction extras
  size_t sc_row = 0, sc_grp = 0;               // int8 activation scales
  size_t widen = 0;                            // int8 weights given as bytes: one projection's operand form
  size_t total = 0;
  int vt_ld = 0;
};

// Activation-scale group of the FC2 input on the int8 path ([linlog]
// "int8 量化": one scale per 1024 FC2 input channels; a block with F <= 1024
// has one group).
int fc2_group(const h3dit_config* c) { return std::min(c->ffn, 1024); }

// Activation arenas aliased by lifetime ([linlog] "DiT 融合内核", activation
// buffer aliasing):  a1 holds Q, K, V^T and then the FC1 output u; a2 holds
// h, then the attention output o, then h2, then the next block's h; a3 holds
// the out-projection output and then the FC2 output.  On the int8 path a2
// holds int8 codes (as BF16 values) instead of h, o and h2 -- the attention
// output goes to a3 and is quantised into a2 -- FC1's output u is quantised
// in place in a1, and two small scale buffers are added: sc_row [N] (the
// per-token scale of whichever projection input is live) and sc_grp
// [N][F / 1024] (the FC2 input's group scales).
Arena plan_arena(const h3dit_config* c, int n, const h3dit_reduction* tr) {
  Arena a;
  const size_t d = c->d, F = c->ffn;
  a.vt_ld = (int)round_up((size_t)n, 64);
  const size_t qk = round_up(n * d * 2, 256);
  const size_t vt = round_up((size_t)c->heads * c->head_dim * a.vt_ld * 2, 256);
  const size_t a1 = std::max(2 * qk + vt, round_up(n * F * 2, 256));
  const size_t nd = round_up(n * d * 2, 256);
  size_t off = 0;
  a.a1 = off; off += a1;
  a.a2 = off; off += nd;
  a.a3 = off; off += nd;
  a.rope = off; off += round_up((size_t)n * (c->head_dim / 2) * 8, 256);
  if (int8_set(c->precision).any()) {
    a.sc_row = off; off += round_up((size_t)n * 4, 256);
    a.sc_grp = off; off += round_up((size_t)n * (F / fc2_group(c)) * 4, 256);
    const Int8Set q8 = int8_set(c->precision);
    size_t wmax = 0;
    if (q8.qkv) wmax = std::max(wmax, 3 * d * d);
    if (q8.o) wmax = std::max(wmax, d * d);
    if (q8.fc1 || q8.fc2) wmax = std::max(wmax, F * d);
    a.widen = off; off += round_up(wmax * 2, 256);
  }
  if (tr) {
    const h3::PairGrid g = pair_grid(&tr->grid, n);
    a.xred = off; off += round_up((size_t)g.n_red * d * 2, 256);
    a.rope_red = off; off += round_up((size_t)g.n_red * (c->head_dim / 2) * 8, 256);
    a.pos_red = off; off += round_up((size_t)g.n_red * 3 * 4, 256);
  }
  a.total = off;
  return a;
}

struct BlockBufs {
  uint8_t* base;
  Arena ar;
};

// One block's sub-steps from its AdaLN-1 output (already in a2) to the final
// gated residual.  Projections in `q8` run on int8 codes ([linlog] "int8
// 量化"): their input is quantised per token (FC2's per token and per 1024
// channels) and a2 then holds codes, with the scales in sc_row / sc_grp;
// the others run in BF16.  Attention stays BF16.  next_shift/next_scale: the
// following block's AdaLN-1 vectors to emit into a2 from the residual
// kernel (as codes if that block's QKV is int8), or NULL.
h3dit_status run_block_body(const h3dit_config* c, const h3dit_block_weights* w, const float* mod, bf16* x,
                            int n, const float* rope, const BlockBufs& B, int vt_ld,
                            const float* next_shift, const float* next_scale, cudaStream_t s,
                            const h3::SegMap& sm) {
  const int d = c->d, F = c->ffn, dh = c->head_dim;
  const Int8Set q8 = int8_set(c->precision);
  const int g2 = fc2_group(c);
  uint8_t* a1 = B.base + B.ar.a1;
  bf16* a2 = reinterpret_cast<bf16*>(B.base + B.ar.a2);
  bf16* a3 = reinterpret_cast<bf16*>(B.base + B.ar.a3);
  float* sc_row = q8.any() ? reinterpret_cast<float*>(B.base + B.ar.sc_row) : nullptr;
  float* sc_grp = q8.any() ? reinterpret_cast<float*>(B.base + B.ar.sc_grp) : nullptr;
  // int8 weights given as bytes are widened into this slot just before
  // their projection (every projection is done with it before the next)
  bf16* slot = q8.any() ? reinterpret_cast<bf16*>(B.base + B.ar.widen) : nullptr;
  auto weight = [&](const void* wq, size_t count, const void** out) -> h3dit_status {
    *out = wq;
    if (!w->codes_int8) return H3DIT_OK;
    TimedLaunch tl(kQuant, s);
    const size_t n8 = count / 8;
    H3_TRY(launch_ex(h3::widen_codes_kernel, dim3((unsigned)((n8 + 255) / 256)), dim3(256), 0, s, 1,
                     static_cast<const int8_t*>(wq), n8, slot));
    *out = slot;
    return H3DIT_OK;
  };
  bf16* q = reinterpret_cast<bf16*>(a1);
  bf16* k = reinterpret_cast<bf16*>(a1 + round_up((size_t)n * d * 2, 256));
  bf16* vt = reinterpret_cast<bf16*>(a1 + 2 * round_up((size_t)n * d * 2, 256));
  bf16* u = reinterpret_cast<bf16*>(a1);
  const float* gate1 = mod + 2 * d;
  const float* shift2 = mod + 3 * d;
  const float* scale2 = mod + 4 * d;
  const float* gate2 = mod + 5 * d;

  h3::GemmArgs g{};
  g.q = q; g.k = k; g.vt = vt; g.vt_ld = vt_ld; g.d = d; g.head_dim = dh;
  g.rope = reinterpret_cast<const float2*>(rope);
  if (q8.qkv) {
    const void* wq;
    H3_TRY(weight(w->w_qkv, (size_t)3 * d * d, &wq));
    H3_TRY(launch_gemm_i8(h3::kEpiQKV, a2, sc_row, d, wq, w->s_qkv, n, 3 * d, d, g, nullptr, kQKV, s));
  } else
    H3_TRY(launch_gemm(h3::kEpiQKV, a2, w->w_qkv, n, 3 * d, d, g, kQKV, s));
  h3::GemmArgs go{};
  go.c = a3; go.ldc = d;
  if (q8.o) {
    // o into a3, its codes into a2 (h is dead), the projection back into a3
    H3_TRY(launch_attention(c, q, k, vt, vt_ld, n, a3, s));
    H3_TRY(launch_quantize_codes(a3, n, d, d, a2, sc_row, s));
    const void* wq;
    H3_TRY(weight(w->w_o, (size_t)d * d, &wq));
    H3_TRY(launch_gemm_i8(h3::kEpiStore, a2, sc_row, d, wq, w->s_o, n, d, d, go, nullptr, kOProj, s));
  } else {
    H3_TRY(launch_attention(c, q, k, vt, vt_ld, n, a2, s));
    H3_TRY(launch_gemm(h3::kEpiStore, a2, w->w_o, n, d, d, go, kOProj, s));
  }
  H3_TRY(launch_rows(x, a3, gate1, shift2, scale2, a2, q8.fc1 ? sc_row : nullptr, n, d, c->eps, s, sm));
  h3::GemmArgs g1{};
  g1.c = u; g1.ldc = F;
  if (q8.fc1) {
    const void* wq;
    H3_TRY(weight(w->w1, (size_t)F * d, &wq));
    H3_TRY(launch_gemm_i8(h3::kEpiGelu, a2, sc_row, d, wq, w->s1, n, F, d, g1, nullptr, kFC1, s));
  } else
    H3_TRY(launch_gemm(h3::kEpiGelu, a2, w->w1, n, F, d, g1, kFC1, s));
  h3::GemmArgs gm{};
  gm.c = a3; gm.ldc = d;
  if (q8.fc2) {
    H3_TRY(launch_quantize_codes(u, n, F, g2, u, sc_grp, s));
    const void* wq;
    H3_TRY(weight(w->w2, (size_t)d * F, &wq));
    H3_TRY(launch_gemm_i8(h3::kEpiStore, u, sc_grp, g2, wq, w->s2, n, d, F, gm, nullptr, kFC2, s));
  } else {
    H3_TRY(launch_gemm(h3::kEpiStore, u, w->w2, n, d, F, gm, kFC2, s));
  }
  H3_TRY(launch_rows(x, a3, gate2, next_shift, next_scale, a2, (next_shift && q8.qkv) ? sc_row : nullptr, n, d,
                     c->eps, s, sm));
  return H3DIT_OK;
}

// The segment map of a modulation table [count][6][d]; NULL segments = one.
h3dit_status make_segmap(const h3dit_segments* seg, int n_tokens, int d, h3::SegMap* out) {
  h3::SegMap m{};
  m.count = 1;
  m.stride = 6 * d;
  if (seg) {
    if (seg->count < 1 || seg->count > 4) return fail(H3DIT_E_INVAL, "segment count %d (1..4)", seg->count);
    if (seg->start[0] != 0) return fail(H3DIT_E_INVAL, "the first segment must start at row 0");
    for (int i = 1; i < seg->count; ++i)
      if (seg->start[i] <= seg->start[i - 1] || seg->start[i] >= n_tokens)
        return fail(H3DIT_E_INVAL, "segment starts must increase and lie inside the %d rows", n_tokens);
    m.count = seg->count;
    for (int i = 0; i < seg->count; ++i) m.start[i] = seg->start[i];
  }
  *out = m;
  return H3DIT_OK;
}

// The segment map of the reduced stream: boundaries before the video grid
// stay, boundaries after it move up by the rows the pairing removed; a
// boundary inside the grid is refused (a pair must lie in one segment).
h3dit_status reduce_segmap(const h3::SegMap& m, const h3::PairGrid& g, h3::SegMap* out) {
  h3::SegMap r = m;
  const int v0 = g.offset, v1 = g.offset + g.T * g.Hh * g.W;
  const int removed = g.n_full - g.n_red;
  for (int i = 1; i < m.count; ++i) {
    if (m.start[i] <= v0) continue;
    if (m.start[i] < v1) return fail(H3DIT_E_INVAL, "segment start %d lies inside the reduced video grid", m.start[i]);
    r.start[i] = m.start[i] - removed;
  }
  *out = r;
  return H3DIT_OK;
}

h3dit_status check_weights(const h3dit_config* c, const h3dit_block_weights* w) {
  if (!w) return fail(H3DIT_E_INVAL, "weights are NULL");
  if (!w->w_qkv || !w->w_o || !w->w1 || !w->w2) return fail(H3DIT_E_INVAL, "a weight pointer is NULL");
  const Int8Set q8 = int8_set(c->precision);
  if ((q8.qkv && !w->s_qkv) || (q8.o && !w->s_o) || (q8.fc1 && !w->s1) || (q8.fc2 && !w->s2))
    return fail(H3DIT_E_INVAL, "an int8 projection needs its weight scales");
  if (w->codes_int8 != 0 && w->codes_int8 != 1) return fail(H3DIT_E_INVAL, "codes_int8 %d (0 or 1)", w->codes_int8);
  if (w->codes_int8 && ((q8.qkv && !aligned(w->w_qkv, 8)) || (q8.o && !aligned(w->w_o, 8)) ||
                        (q8.fc1 && !aligned(w->w1, 8)) || (q8.fc2 && !aligned(w->w2, 8))))
    return fail(H3DIT_E_INVAL, "int8 weight bytes must be 8-byte aligned");
  return H3DIT_OK;
}

}  // namespace

// ====================================================================== C ABI
extern "C" {

const char* h3dit_last_error(void) { return t_last_error.c_str(); }

int h3dit_version(void) { return H3DIT_VERSION; }

h3dit_status h3dit_check_device_error(cudaStream_t stream) {
  H3_CUDA(cudaStreamSynchronize(stream));
  unsigned int v = 0, zero = 0;
  H3_CUDA(cudaMemcpyFromSymbol(&v, h3::g_device_error, sizeof(v)));
  if (v) {
    H3_CUDA(cudaMemcpyToSymbol(h3::g_device_error, &zero, sizeof(zero)));
    return fail(H3DIT_E_TIMEOUT, "a kernel's pipeline wait ran out of time (device error word 0x%x)", v);
  }
  return H3DIT_OK;
}

h3dit_status h3dit_test_set_wait_limit(unsigned long long ns) {
  const unsigned long long v = ns ? ns : h3::kWaitLimitNs;
  H3_CUDA(cudaMemcpyToSymbol(h3::g_wait_limit_ns, &v, sizeof(v)));
  return H3DIT_OK;
}

h3dit_status h3dit_test_stall_next_gemm(int kblock) {
  if (kblock < -1) return fail(H3DIT_E_INVAL, "kblock %d", kblock);
  g_stall_request.store(kblock);
  return H3DIT_OK;
}

h3dit_status h3dit_timing_enable(int on) {
  std::lock_guard<std::mutex> lk(g_timing.mu);
  g_timing.enabled = on != 0;
  return H3DIT_OK;
}

h3dit_status h3dit_timing_reset(void) {
  std::lock_guard<std::mutex> lk(g_timing.mu);
  for (auto& p : g_timing.pending) {
    cudaEventSynchronize(p.b);
    cudaEventDestroy(p.a);
    cudaEventDestroy(p.b);
  }
  g_timing.pending.clear();
  for (int i = 0; i < kNumClasses; ++i) { g_timing.total_ms[i] = 0; g_timing.count[i] = 0; }
  return H3DIT_OK;
}

h3dit_status h3dit_timing_read(int cls, double* total_ms, long long* launches) {
  if (cls < 0 || cls >= kNumClasses || !total_ms || !launches) return fail(H3DIT_E_INVAL, "bad timing query");
  std::lock_guard<std::mutex> lk(g_timing.mu);
  for (auto& p : g_timing.pending) {
    H3_CUDA(cudaEventSynchronize(p.b));
    float ms = 0.f;
    H3_CUDA(cudaEventElapsedTime(&ms, p.a, p.b));
    g_timing.total_ms[p.cls] += ms;
    g_timing.count[p.cls] += p.kernels;
    cudaEventDestroy(p.a);
    cudaEventDestroy(p.b);
  }
  g_timing.pending.clear();
  *total_ms = g_timing.total_ms[cls];
  *launches = g_timing.count[cls];
  return H3DIT_OK;
}

h3dit_status h3dit_workspace_size(const h3dit_config* cfg, int n_tokens, const h3dit_reduction* tr,
                                  size_t* bytes) {
  H3_TRY(check_cfg(cfg));
  if (!bytes) return fail(H3DIT_E_INVAL, "bytes is NULL");
  if (n_tokens < 1) return fail(H3DIT_E_INVAL, "n_tokens %d", n_tokens);
  if (tr) H3_TRY(check_grid(&tr->grid, n_tokens));
  *bytes = plan_arena(cfg, n_tokens, tr).total;
  return H3DIT_OK;
}

h3dit_status h3dit_rope_table(const h3dit_config* cfg, const float* pos, int n_tokens, float* table,
                              cudaStream_t stream) {
  H3_TRY(check_cfg(cfg));
  if (!pos || !table) return fail(H3DIT_E_INVAL, "NULL pointer");
  if (n_tokens < 1) return fail(H3DIT_E_INVAL, "n_tokens %d", n_tokens);
  return launch_rope_table(cfg, pos, n_tokens, table, stream);
}

h3dit_status h3dit_adaln(const h3dit_config* cfg, const void* x, const float* shift, const float* scale,
                         int n_tokens, void* h, cudaStream_t stream) {
  H3_TRY(check_cfg(cfg));
  if (!x || !shift || !scale || !h) return fail(H3DIT_E_INVAL, "NULL pointer");
  if (n_tokens < 1) return fail(H3DIT_E_INVAL, "n_tokens %d", n_tokens);
  return launch_rows(const_cast<void*>(x), nullptr, nullptr, shift, scale, h, nullptr, n_tokens, cfg->d, cfg->eps,
                     stream);
}

h3dit_status h3dit_gate_residual_adaln(const h3dit_config* cfg, void* x, const void* branch, const float* gate,
                                       const float* shift, const float* scale, int n_tokens, void* h,
                                       cudaStream_t stream) {
  H3_TRY(check_cfg(cfg));
  if (!x || !branch || !gate) return fail(H3DIT_E_INVAL, "NULL pointer");
  if ((shift == nullptr) != (scale == nullptr)) return fail(H3DIT_E_INVAL, "shift and scale must both be set or NULL");
  if (shift && !h) return fail(H3DIT_E_INVAL, "h is NULL");
  if (n_tokens < 1) return fail(H3DIT_E_INVAL, "n_tokens %d", n_tokens);
  return launch_rows(x, branch, gate, shift, scale, h, nullptr, n_tokens, cfg->d, cfg->eps, stream);
}

h3dit_status h3dit_qkv_project(const h3dit_config* cfg, const void* h, const void* w_qkv, const float* table,
                               int n_tokens, void* q, void* k, void* vt, int vt_ld, cudaStream_t stream) {
  H3_TRY(check_cfg(cfg));
  if (!h || !w_qkv || !table || !q || !k || !vt) return fail(H3DIT_E_INVAL, "NULL pointer");
  if (n_tokens < 1) return fail(H3DIT_E_INVAL, "n_tokens %d", n_tokens);
  if (vt_ld < n_tokens || vt_ld % 8 != 0) return fail(H3DIT_E_INVAL, "vt_ld %d", vt_ld);
  if (!aligned(table, 16) || !aligned(q, 16) || !aligned(k, 16) || !aligned(vt, 16))
    return fail(H3DIT_E_INVAL, "outputs must be 16-byte aligned");
  h3::GemmArgs g{};
  g.q = static_cast<bf16*>(q);
  g.k = static_cast<bf16*>(k);
  g.vt = static_cast<bf16*>(vt);
  g.vt_ld = vt_ld;
  g.d = cfg->d;
  g.head_dim = cfg->head_dim;
  g.rope = reinterpret_cast<const float2*>(table);
  return launch_gemm(h3::kEpiQKV, h, w_qkv, n_tokens, 3 * cfg->d, cfg->d, g, kQKV, stream);
}

h3dit_status h3dit_attention(const h3dit_config* cfg, const void* q, const void* k, const void* vt, int vt_ld,
                             int n_tokens, void* o, cudaStream_t stream) {
  H3_TRY(check_heads(cfg));
  if (!q || !k || !vt || !o) return fail(H3DIT_E_INVAL, "NULL pointer");
  if (n_tokens < 1) return fail(H3DIT_E_INVAL, "n_tokens %d", n_tokens);
  return launch_attention(cfg, q, k, vt, vt_ld, n_tokens, o, stream);
}

h3dit_status h3dit_linear(const void* a, const void* b, int m, int n, int k, int act, void* c,
                          cudaStream_t stream) {
  if (!a || !b || !c) return fail(H3DIT_E_INVAL, "NULL pointer");
  if (m < 1 || n < 1 || k < 1) return fail(H3DIT_E_INVAL, "non-positive shape");
  if (act != 0 && act != 1) return fail(H3DIT_E_INVAL, "act %d", act);
  if (!aligned(c, 16)) return fail(H3DIT_E_INVAL, "c must be 16-byte aligned");
  h3::GemmArgs g{};
  g.c = static_cast<bf16*>(c);
  g.ldc = n;
  return launch_gemm(act ? h3::kEpiGelu : h3::kEpiStore, a, b, m, n, k, g, act ? kFC1 : kOProj, stream);
}

static h3dit_status block_forward_impl(const h3dit_config* cfg, const h3dit_block_weights* w, const float* mod,
                                const h3dit_segments* seg, void* x, const float* pos, int n_tokens, void* ws,
                                size_t ws_bytes, cudaStream_t stream) {
  H3_TRY(check_cfg(cfg));
  const FaultKind fk = injected_fault();
  if (fk == kFaultShape) return fail(H3DIT_E_UNSUPPORTED, "injected unsupported shape (H3DIT_FAULT=shape)");
  H3_TRY(check_weights(cfg, w));
  if (!mod || !x || !pos || !ws) return fail(H3DIT_E_INVAL, "NULL pointer");
  if (fk == kFaultArg) return fail(H3DIT_E_INVAL, "injected invalid argument (H3DIT_FAULT=arg)");
  if (n_tokens < 1) return fail(H3DIT_E_INVAL, "n_tokens %d", n_tokens);
  if (!aligned(ws, 256) || !aligned(x, 16)) return fail(H3DIT_E_INVAL, "ws must be 256-byte and x 16-byte aligned");
  h3::SegMap sm;
  H3_TRY(make_segmap(seg, n_tokens, cfg->d, &sm));
  const Arena ar = plan_arena(cfg, n_tokens, nullptr);
  if (ws_bytes < ar.total || fk == kFaultAlloc)
    return fail(H3DIT_E_NOMEM, "workspace %zu < %zu bytes%s", ws_bytes, ar.total,
                fk == kFaultAlloc ? " (injected: H3DIT_FAULT=alloc)" : "");
  BlockBufs B{static_cast<uint8_t*>(ws), ar};
  float* rope = reinterpret_cast<float*>(B.base + ar.rope);
  bf16* xb = static_cast<bf16*>(x);
  const int d = cfg->d;
  NvtxRange trace("h3dit block");
  H3_TRY(launch_rope_table(cfg, pos, n_tokens, rope, stream));
  float* hs = int8_set(cfg->precision).qkv ? reinterpret_cast<float*>(B.base + ar.sc_row) : nullptr;
  H3_TRY(launch_rows(xb, nullptr, nullptr, mod + 0 * d, mod + 1 * d, B.base + ar.a2, hs, n_tokens, d, cfg->eps,
                     stream, sm));
  return run_block_body(cfg, w, mod, xb, n_tokens, rope, B, ar.vt_ld, nullptr, nullptr, stream, sm);
}

static h3dit_status step_forward_impl(const h3dit_config* cfg, const h3dit_block_weights* w, int n_blocks,
                               const float* mods, const h3dit_segments* seg, void* x, const float* pos, int n_tokens,
                               const h3dit_reduction* tr, void* ws, size_t ws_bytes, cudaStream_t stream) {
  H3_TRY(check_cfg(cfg));
  const FaultKind fk = injected_fault();
  if (fk == kFaultShape) return fail(H3DIT_E_UNSUPPORTED, "injected unsupported shape (H3DIT_FAULT=shape)");
  if (!w || n_blocks < 0) return fail(H3DIT_E_INVAL, "weights NULL or n_blocks < 0");
  if (n_blocks == 0) return H3DIT_OK;
  for (int b = 0; b < n_blocks; ++b) H3_TRY(check_weights(cfg, &w[b]));
  if (!mods || !x || !pos || !ws) return fail(H3DIT_E_INVAL, "NULL pointer");
  if (fk == kFaultArg) return fail(H3DIT_E_INVAL, "injected invalid argument (H3DIT_FAULT=arg)");
  if (n_tokens < 1) return fail(H3DIT_E_INVAL, "n_tokens %d", n_tokens);
  if (!aligned(ws, 256) || !aligned(x, 16)) return fail(H3DIT_E_INVAL, "ws must be 256-byte and x 16-byte aligned");
  if (tr) {
    H3_TRY(check_grid(&tr->grid, n_tokens));
    if (tr->reduce_after_block < 0 || tr->restore_before_block <= tr->reduce_after_block)
      return fail(H3DIT_E_INVAL, "reduction blocks %d / %d", tr->reduce_after_block, tr->restore_before_block);
  }
  h3::SegMap sm_full;
  H3_TRY(make_segmap(seg, n_tokens, cfg->d, &sm_full));
  h3::SegMap sm_red = sm_full;
  if (tr) H3_TRY(reduce_segmap(sm_full, pair_grid(&tr->grid, n_tokens), &sm_red));
  const size_t per_block = (size_t)sm_full.count * 6 * cfg->d;   // modulation floats per block
  const Arena ar = plan_arena(cfg, n_tokens, tr);
  if (ws_bytes < ar.total || fk == kFaultAlloc)
    return fail(H3DIT_E_NOMEM, "workspace %zu < %zu bytes%s", ws_bytes, ar.total,
                fk == kFaultAlloc ? " (injected: H3DIT_FAULT=alloc)" : "");
  BlockBufs B{static_cast<uint8_t*>(ws), ar};
  const int d = cfg->d;
  bf16* xfull = static_cast<bf16*>(x);
  float* rope_full = reinterpret_cast<float*>(B.base + ar.rope);
  NvtxRange trace("h3dit step");
  H3_TRY(launch_rope_table(cfg, pos, n_tokens, rope_full, stream));

  h3::PairGrid pg{};
  bf16* xred = nullptr;
  float* rope_red = nullptr;
  if (tr) {
    pg = pair_grid(&tr->grid, n_tokens);
    xred = reinterpret_cast<bf16*>(B.base + ar.xred);
    rope_red = reinterpret_cast<float*>(B.base + ar.rope_red);
    const float* pr = tr->pos_reduced;
    if (!pr) {
      float* p = reinterpret_cast<float*>(B.base + ar.pos_red);
      TimedLaunch tl(kReduce, stream);
      h3::reduced_positions_kernel<<<(pg.n_red + 127) / 128, 128, 0, stream>>>(pos, pg, p);
      H3_CUDA(cudaGetLastError());
      pr = p;
    }
    H3_TRY(launch_rope_table(cfg, pr, pg.n_red, rope_red, stream));
  }

  bf16* cur = xfull;
  int cur_n = n_tokens;
  const float* cur_rope = rope_full;
  bool reduced = false;
  float* hs = int8_set(cfg->precision).qkv ? reinterpret_cast<float*>(B.base + ar.sc_row) : nullptr;
  const h3::SegMap* cur_sm = &sm_full;
  H3_TRY(launch_rows(cur, nullptr, nullptr, mods, mods + d, B.base + ar.a2, hs, cur_n, d, cfg->eps, stream, *cur_sm));
  for (int b = 0; b < n_blocks; ++b) {
    const float* mod = mods + per_block * b;
    const bool last = b + 1 == n_blocks;
    const bool reduce_now = tr && !reduced && b == tr->reduce_after_block && b + 1 < tr->restore_before_block && !last;
    const bool restore_now = tr && reduced && b + 1 == tr->restore_before_block && !last;
    const float* nmod = last ? nullptr : mods + per_block * (b + 1);
    const bool emit_next = !last && !reduce_now && !restore_now;
    const int vt_ld = (int)round_up((size_t)cur_n, 64);
    NvtxRange block_trace("h3dit block", b);
    H3_TRY(run_block_body(cfg, &w[b], mod, cur, cur_n, cur_rope, B, vt_ld,
                          emit_next ? nmod : nullptr, emit_next ? nmod + d : nullptr, stream, *cur_sm));
    if (reduce_now) {
      {
        TimedLaunch tl(kReduce, stream);
        h3::token_reduce_kernel<<<pg.n_red, h3::kRowThreads, 0, stream>>>(xfull, d, pg, xred, nullptr);
        H3_CUDA(cudaGetLastError());
      }
      cur = xred;
      cur_n = pg.n_red;
      cur_rope = rope_red;
      reduced = true;
      cur_sm = &sm_red;
      H3_TRY(launch_rows(cur, nullptr, nullptr, nmod, nmod + d, B.base + ar.a2, hs, cur_n, d, cfg->eps, stream,
                         *cur_sm));
    } else if (restore_now) {
      {
        TimedLaunch tl(kReduce, stream);
        h3::token_restore_kernel<<<pg.n_red, h3::kRowThreads, 0, stream>>>(xred, xfull, d, pg, xfull);
        H3_CUDA(cudaGetLastError());
      }
      cur = xfull;
      cur_n = n_tokens;
      cur_rope = rope_full;
      reduced = false;
      cur_sm = &sm_full;
      H3_TRY(launch_rows(cur, nullptr, nullptr, nmod, nmod + d, B.base + ar.a2, hs, cur_n, d, cfg->eps, stream,
                         *cur_sm));
    }
  }
  if (reduced) {
    TimedLaunch tl(kReduce, stream);
    h3::token_restore_kernel<<<pg.n_red, h3::kRowThreads, 0, stream>>>(xred, xfull, d, pg, xfull);
    H3_CUDA(cudaGetLastError());
  }
  return H3DIT_OK;
}

h3dit_status h3dit_block_forward(const h3dit_config* cfg, const h3dit_block_weights* w, const float* mod,
                                 void* x, const float* pos, int n_tokens, void* ws, size_t ws_bytes,
                                 cudaStream_t stream) {
  return block_forward_impl(cfg, w, mod, nullptr, x, pos, n_tokens, ws, ws_bytes, stream);
}

h3dit_status h3dit_block_forward_seg(const h3dit_config* cfg, const h3dit_block_weights* w, const float* mods,
                                     const h3dit_segments* seg, void* x, const float* pos, int n_tokens, void* ws,
                                     size_t ws_bytes, cudaStream_t stream) {
  if (!seg) return fail(H3DIT_E_INVAL, "segments are NULL");
  return block_forward_impl(cfg, w, mods, seg, x, pos, n_tokens, ws, ws_bytes, stream);
}

h3dit_status h3dit_step_forward(const h3dit_config* cfg, const h3dit_block_weights* w, int n_blocks,
                                const float* mods, void* x, const float* pos, int n_tokens,
                                const h3dit_reduction* tr, void* ws, size_t ws_bytes, cudaStream_t stream) {
  return step_forward_impl(cfg, w, n_blocks, mods, nullptr, x, pos, n_tokens, tr, ws, ws_bytes, stream);
}

h3dit_status h3dit_step_forward_seg(const h3dit_config* cfg, const h3dit_block_weights* w, int n_blocks,
                                    const float* mods, const h3dit_segments* seg, void* x, const float* pos,
                                    int n_tokens, const h3dit_reduction* tr, void* ws, size_t ws_bytes,
                                    cudaStream_t stream) {
  if (!seg) return fail(H3DIT_E_INVAL, "segments are NULL");
  return step_forward_impl(cfg, w, n_blocks, mods, seg, x, pos, n_tokens, tr, ws, ws_bytes, stream);
}

h3dit_status h3dit_quantize_act(const void* x_bf16, int rows, int cols, int group, int8_t* q, float* scales,
                                cudaStream_t stream) {
  if (!x_bf16 || !q || !scales) return fail(H3DIT_E_INVAL, "NULL pointer");
  if (rows < 1 || cols < 1 || group < 1) return fail(H3DIT_E_INVAL, "non-positive shape");
  if (cols % group != 0) return fail(H3DIT_E_INVAL, "group %d does not divide cols %d", group, cols);
  if (group % 8 != 0) return fail(H3DIT_E_UNSUPPORTED, "group %d (multiple of 8)", group);
  if (!aligned(x_bf16, 16) || !aligned(q, 8)) return fail(H3DIT_E_INVAL, "x must be 16-byte, q 8-byte aligned");
  const long long blocks = 1LL * rows * (cols / group);
  if (blocks > 0x7fffffffLL) return fail(H3DIT_E_UNSUPPORTED, "too many groups");
  TimedLaunch tl(kQuant, stream);
  bool done = false;
  H3_TRY(launch_quantize_warp<false>(x_bf16, rows, cols, group, nullptr, q, scales, stream, &done));
  if (!done)
    h3::quantize_kernel<<<(unsigned)blocks, h3::kRowThreads, 0, stream>>>(static_cast<const bf16*>(x_bf16), cols, group,
                                                                         q, scales);
  H3_CUDA(cudaGetLastError());
  return H3DIT_OK;
}

h3dit_status h3dit_quantize_weight(const void* w_bf16, int out, int in, int8_t* q, float* scales,
                                   cudaStream_t stream) {
  return h3dit_quantize_act(w_bf16, out, in, in, q, scales, stream);
}

h3dit_status h3dit_quantize_codes(const void* x_bf16, int rows, int cols, int group, void* q_bf16, float* scales,
                                  cudaStream_t stream) {
  if (!x_bf16 || !q_bf16 || !scales) return fail(H3DIT_E_INVAL, "NULL pointer");
  if (rows < 1 || cols < 1 || group < 1) return fail(H3DIT_E_INVAL, "non-positive shape");
  if (cols % group != 0) return fail(H3DIT_E_INVAL, "group %d does not divide cols %d", group, cols);
  if (group % 8 != 0) return fail(H3DIT_E_UNSUPPORTED, "group %d (multiple of 8)", group);
  if (!aligned(x_bf16, 16) || !aligned(q_bf16, 16)) return fail(H3DIT_E_INVAL, "x and q must be 16-byte aligned");
  return launch_quantize_codes(x_bf16, rows, cols, group, q_bf16, scales, stream);
}

h3dit_status h3dit_widen_codes(const int8_t* q, size_t count, void* q_bf16, cudaStream_t stream) {
  if (!q || !q_bf16) return fail(H3DIT_E_INVAL, "NULL pointer");
  if (count == 0) return H3DIT_OK;
  if (count % 8 != 0) return fail(H3DIT_E_UNSUPPORTED, "count %zu (multiple of 8)", count);
  if (!aligned(q, 8) || !aligned(q_bf16, 16)) return fail(H3DIT_E_INVAL, "q must be 8-byte, q_bf16 16-byte aligned");
  const size_t n8 = count / 8;
  const size_t blocks = (n8 + 255) / 256;
  if (blocks > 0x7fffffffULL) return fail(H3DIT_E_UNSUPPORTED, "count %zu too large", count);
  TimedLaunch tl(kQuant, stream);
  h3::widen_codes_kernel<<<(unsigned)blocks, 256, 0, stream>>>(q, n8, static_cast<bf16*>(q_bf16));
  H3_CUDA(cudaGetLastError());
  return H3DIT_OK;
}

h3dit_status h3dit_adaln_quant(const h3dit_config* cfg, const void* x, const float* shift, const float* scale,
                               int n_tokens, void* hq, float* hs, cudaStream_t stream) {
  H3_TRY(check_cfg(cfg));
  if (!x || !shift || !scale || !hq || !hs) return fail(H3DIT_E_INVAL, "NULL pointer");
  if (n_tokens < 1) return fail(H3DIT_E_INVAL, "n_tokens %d", n_tokens);
  return launch_rows(const_cast<void*>(x), nullptr, nullptr, shift, scale, hq, hs, n_tokens, cfg->d, cfg->eps,
                     stream);
}

h3dit_status h3dit_gate_residual_adaln_quant(const h3dit_config* cfg, void* x, const void* branch, const float* gate,
                                             const float* shift, const float* scale, int n_tokens, void* hq,
                                             float* hs, cudaStream_t stream) {
  H3_TRY(check_cfg(cfg));
  if (!x || !branch || !gate || !shift || !scale || !hq || !hs) return fail(H3DIT_E_INVAL, "NULL pointer");
  if (n_tokens < 1) return fail(H3DIT_E_INVAL, "n_tokens %d", n_tokens);
  return launch_rows(x, branch, gate, shift, scale, hq, hs, n_tokens, cfg->d, cfg->eps, stream);
}

h3dit_status h3dit_linear_i8(const void* a_codes, const float* sa, int group, const void* b_codes, const float* sb,
                             int m, int n, int k, int act, void* c, cudaStream_t stream) {
  if (!a_codes || !sa || !b_codes || !sb || !c) return fail(H3DIT_E_INVAL, "NULL pointer");
  if (m < 1 || n < 1 || k < 1) return fail(H3DIT_E_INVAL, "non-positive shape");
  if (act != 0 && act != 1) return fail(H3DIT_E_INVAL, "act %d", act);
  if (group < 1 || group > k) return fail(H3DIT_E_INVAL, "group %d (1..k)", group);
  if (!aligned(c, 16)) return fail(H3DIT_E_INVAL, "c must be 16-byte aligned");
  h3::GemmArgs g{};
  g.c = static_cast<bf16*>(c);
  g.ldc = n;
  return launch_gemm_i8(act ? h3::kEpiGelu : h3::kEpiStore, a_codes, sa, group, b_codes, sb, m, n, k, g, nullptr,
                        act ? kFC1 : kOProj, stream);
}

h3dit_status h3dit_linear_i8_acc(const void* a_codes, const void* b_codes, int m, int n, int k, int32_t* acc,
                                 cudaStream_t stream) {
  if (!a_codes || !b_codes || !acc) return fail(H3DIT_E_INVAL, "NULL pointer");
  if (m < 1 || n < 1 || k < 1) return fail(H3DIT_E_INVAL, "non-positive shape");
  if (!aligned(acc, 16)) return fail(H3DIT_E_INVAL, "acc must be 16-byte aligned");
  h3::GemmArgs g{};
  return launch_gemm_i8(h3::kEpiAcc, a_codes, nullptr, k, b_codes, nullptr, m, n, k, g, acc, kOProj, stream);
}

h3dit_status h3dit_qkv_project_i8(const h3dit_config* cfg, const void* hq, const float* hs, const void* w_qkv,
                                  const float* s_qkv, const float* table, int n_tokens, void* q, void* k, void* vt,
                                  int vt_ld, cudaStream_t stream) {
  H3_TRY(check_cfg(cfg));
  if (!hq || !hs || !w_qkv || !s_qkv || !table || !q || !k || !vt) return fail(H3DIT_E_INVAL, "NULL pointer");
  if (n_tokens < 1) return fail(H3DIT_E_INVAL, "n_tokens %d", n_tokens);
  if (vt_ld < n_tokens || vt_ld % 8 != 0) return fail(H3DIT_E_INVAL, "vt_ld %d", vt_ld);
  if (!aligned(table, 16) || !aligned(q, 16) || !aligned(k, 16) || !aligned(vt, 16))
    return fail(H3DIT_E_INVAL, "outputs must be 16-byte aligned");
  h3::GemmArgs g{};
  g.q = static_cast<bf16*>(q);
  g.k = static_cast<bf16*>(k);
  g.vt = static_cast<bf16*>(vt);
  g.vt_ld = vt_ld;
  g.d = cfg->d;
  g.head_dim = cfg->head_dim;
  g.rope = reinterpret_cast<const float2*>(table);
  return launch_gemm_i8(h3::kEpiQKV, hq, hs, cfg->d, w_qkv, s_qkv, n_tokens, 3 * cfg->d, cfg->d, g, nullptr, kQKV,
                        stream);
}

h3dit_status h3dit_final_layer(const h3dit_config* cfg, const void* x, int n_tokens, const h3dit_final_head* heads,
                               int n_heads, cudaStream_t stream) {
  H3_TRY(check_cfg(cfg));
  if (!x || !heads) return fail(H3DIT_E_INVAL, "NULL pointer");
  if (n_tokens < 1) return fail(H3DIT_E_INVAL, "n_tokens %d", n_tokens);
  if (n_heads < 1 || n_heads > 4) return fail(H3DIT_E_INVAL, "n_heads %d (1..4)", n_heads);
  if (!aligned(x, 16)) return fail(H3DIT_E_INVAL, "x must be 16-byte aligned");
  const int d = cfg->d;
  for (int i = 0; i < n_heads; ++i) {
    const h3dit_final_head& h = heads[i];
    if (!h.shift || !h.scale || !h.w || !h.out) return fail(H3DIT_E_INVAL, "head %d has a NULL pointer", i);
    if (h.rows < 1 || h.row_start < 0 || h.row_start + h.rows > n_tokens)
      return fail(H3DIT_E_INVAL, "head %d rows %d..%d outside the %d tokens", i, h.row_start, h.row_start + h.rows,
                  n_tokens);
    if (h.c_out < 16 || h.c_out > h3::kHeadMaxN || h.c_out % 16 != 0)
      return fail(H3DIT_E_UNSUPPORTED, "head %d c_out %d (a multiple of 16, 16..256)", i, h.c_out);
    if (!aligned(h.w, 16) || !aligned(h.out, 16) || !aligned(h.shift, 16) || !aligned(h.scale, 16))
      return fail(H3DIT_E_INVAL, "head %d tensors must be 16-byte aligned", i);
  }
  H3_TRY(set_smem(h3::final_head_kernel, h3::head_smem_max()));
  h3::HeadBatch hb{};
  {
    const uint64_t dims[2] = {(uint64_t)d, (uint64_t)n_tokens};
    const uint64_t str[1] = {(uint64_t)d * 2};
    const uint32_t box[2] = {h3::kHeadBK, 128};
    H3_TRY(make_map(&hb.tmX, x, 2, dims, str, box));
  }
  int max_tiles = 0, all_tiles = 0;
  size_t smem = 0;
  h3::HeadRows hr{};
  hr.n_heads = n_heads;
  for (int i = 0; i < n_heads; ++i) {
    const h3dit_final_head& h = heads[i];
    const uint64_t dims[2] = {(uint64_t)d, (uint64_t)h.c_out};
    const uint64_t str[1] = {(uint64_t)d * 2};
    const uint32_t box[2] = {h3::kHeadBK, (uint32_t)h.c_out};
    H3_TRY(make_map(&hb.tmW[i], h.w, 2, dims, str, box));
    h3::HeadArgs& a = hb.a[i];
    a.row_start = h.row_start;
    a.rows = h.rows;
    a.d = d;
    a.shift = h.shift;
    a.scale = h.scale;
    a.c_out = h.c_out;
    a.out = static_cast<bf16*>(h.out);
    uint32_t cols = 32;
    while (cols < (uint32_t)h.c_out) cols <<= 1;
    a.tmem_cols = cols;
    a.stages = h3::head_stages(h.c_out);
    if ((size_t)a.stages * h3::head_stage_bytes(h.c_out) < h3::head_part_bytes(h.c_out))
      return fail(H3DIT_E_UNSUPPORTED, "head %d: c_out %d partial sums exceed the stage ring", i, h.c_out);
    max_tiles = std::max(max_tiles, (h.rows + 127) / 128);
    all_tiles += (h.rows + 127) / 128;
    smem = std::max(smem, h3::head_smem_bytes(h.c_out));
    hr.first_warp[i + 1] = hr.first_warp[i] + h.rows;
    hr.row_start[i] = h.row_start;
    hr.c_out[i] = h.c_out;
    hr.out[i] = static_cast<bf16*>(h.out);
  }
  // split d over a cluster of CTAs so the launch fills the SMs (one wave:
  // every cluster of a tile must fit at once)
  int ksplit = std::max(1, std::min(h3::kHeadMaxSplit, sm_count() / all_tiles));
  ksplit = std::min(ksplit, d / h3::kHeadBK);
  hb.ksplit = ksplit;
  TimedLaunch tl(kRows, stream);
  tl.kernels = 2;   // statistics, then the heads
  const long long stat_threads = (long long)hr.first_warp[n_heads] * 32;
  H3_TRY(launch_ex(h3::head_stats_kernel, dim3((unsigned)((stat_threads + 255) / 256)), dim3(256), 0, stream, 1,
                   static_cast<const bf16*>(x), hr, d, cfg->eps));
  cudaLaunchConfig_t lc{};
  lc.gridDim = dim3(max_tiles * ksplit, n_heads);
  lc.blockDim = dim3(h3::kHeadThreads);
  lc.dynamicSmemBytes = smem;
  lc.stream = stream;
  cudaLaunchAttribute attr[2];
  int na = 0;
  if (ksplit > 1) {
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = ksplit;
    attr[na].val.clusterDim.y = 1;
    attr[na].val.clusterDim.z = 1;
    ++na;
  }
  // the head kernel's x loads overlap the statistics launch's tail; its
  // transform warps wait for that launch before reading the statistics
  if (pdl_enabled()) {
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  lc.attrs = attr;
  lc.numAttrs = na;
  H3_CUDA(cudaLaunchKernelEx(&lc, h3::final_head_kernel, hb));
  return H3DIT_OK;
}

h3dit_status h3dit_core_residual(const void* x_in, const void* x_out, size_t count, float* delta,
                                 cudaStream_t stream) {
  if (!x_in || !x_out || !delta) return fail(H3DIT_E_INVAL, "NULL pointer");
  if (count == 0) return H3DIT_OK;
  if (count % 8 != 0) return fail(H3DIT_E_UNSUPPORTED, "count %zu (multiple of 8)", count);
  if (!aligned(x_in, 16) || !aligned(x_out, 16) || !aligned(delta, 16))
    return fail(H3DIT_E_INVAL, "tensors must be 16-byte aligned");
  const size_t n8 = count / 8, blocks = (n8 + 255) / 256;
  if (blocks > 0x7fffffffULL) return fail(H3DIT_E_UNSUPPORTED, "count %zu too large", count);
  TimedLaunch tl(kRows, stream);
  h3::core_residual_kernel<<<(unsigned)blocks, 256, 0, stream>>>(static_cast<const bf16*>(x_in),
                                                                  static_cast<const bf16*>(x_out), n8, delta);
  H3_CUDA(cudaGetLastError());
  return H3DIT_OK;
}

h3dit_status h3dit_core_reuse(void* x, const float* delta, size_t count, cudaStream_t stream) {
  if (!x || !delta) return fail(H3DIT_E_INVAL, "NULL pointer");
  if (count == 0) return H3DIT_OK;
  if (count % 8 != 0) return fail(H3DIT_E_UNSUPPORTED, "count %zu (multiple of 8)", count);
  if (!aligned(x, 16) || !aligned(delta, 16)) return fail(H3DIT_E_INVAL, "tensors must be 16-byte aligned");
  const size_t n8 = count / 8, blocks = (n8 + 255) / 256;
  if (blocks > 0x7fffffffULL) return fail(H3DIT_E_UNSUPPORTED, "count %zu too large", count);
  TimedLaunch tl(kRows, stream);
  h3::core_reuse_kernel<<<(unsigned)blocks, 256, 0, stream>>>(static_cast<bf16*>(x), delta, n8);
  H3_CUDA(cudaGetLastError());
  return H3DIT_OK;
}

int h3dit_reduced_tokens(int n_tokens, const h3dit_video_grid* g) {
  if (!g || check_grid(g, n_tokens) != H3DIT_OK) return -1;
  return pair_grid(g, n_tokens).n_red;
}

h3dit_status h3dit_token_reduce(const void* x_full, int n_tokens, int d, const h3dit_video_grid* grid, void* x_red,
                                void* side, cudaStream_t stream) {
  if (!x_full || !x_red) return fail(H3DIT_E_INVAL, "NULL pointer");
  if (n_tokens < 1 || d < 8 || d % 8 != 0) return fail(H3DIT_E_INVAL, "shape %d x %d (d %% 8 == 0)", n_tokens, d);
  H3_TRY(check_grid(grid, n_tokens));
  if (!aligned(x_full, 16) || !aligned(x_red, 16) || (side && !aligned(side, 16)))
    return fail(H3DIT_E_INVAL, "tensors must be 16-byte aligned");
  const h3::PairGrid pg = pair_grid(grid, n_tokens);
  TimedLaunch tl(kReduce, stream);
  h3::token_reduce_kernel<<<pg.n_red, h3::kRowThreads, 0, stream>>>(static_cast<const bf16*>(x_full), d, pg,
                                                                    static_cast<bf16*>(x_red), static_cast<bf16*>(side));
  H3_CUDA(cudaGetLastError());
  return H3DIT_OK;
}

h3dit_status h3dit_token_restore(const void* x_red, const void* side, int n_tokens, int d,
                                 const h3dit_video_grid* grid, void* x_full, cudaStream_t stream) {
  if (!x_red || !side || !x_full) return fail(H3DIT_E_INVAL, "NULL pointer");
  if (n_tokens < 1 || d < 8 || d % 8 != 0) return fail(H3DIT_E_INVAL, "shape %d x %d (d %% 8 == 0)", n_tokens, d);
  H3_TRY(check_grid(grid, n_tokens));
  if (!aligned(x_full, 16) || !aligned(x_red, 16) || !aligned(side, 16))
    return fail(H3DIT_E_INVAL, "tensors must be 16-byte aligned");
  const h3::PairGrid pg = pair_grid(grid, n_tokens);
  TimedLaunch tl(kReduce, stream);
  h3::token_restore_kernel<<<pg.n_red, h3::kRowThreads, 0, stream>>>(
      static_cast<const bf16*>(x_red), static_cast<const bf16*>(side), d, pg, static_cast<bf16*>(x_full));
  H3_CUDA(cudaGetLastError());
  return H3DIT_OK;
}

h3dit_status h3dit_reduced_positions(const float* pos, int n_tokens, const h3dit_video_grid* grid, float* pos_red,
                                     cudaStream_t stream) {
  if (!pos || !pos_red) return fail(H3DIT_E_INVAL, "NULL pointer");
  if (n_tokens < 1) return fail(H3DIT_E_INVAL, "n_tokens %d", n_tokens);
  H3_TRY(check_grid(grid, n_tokens));
  const h3::PairGrid pg = pair_grid(grid, n_tokens);
  TimedLaunch tl(kReduce, stream);
  h3::reduced_positions_kernel<<<(pg.n_red + 127) / 128, 128, 0, stream>>>(pos, pg, pos_red);
  H3_CUDA(cudaGetLastError());
  return H3DIT_OK;
}

}  // extern "C"

// ====================================================================== allocation-free block
// Some callers cannot hand the library a workspace: a host program whose
// device memory is owned by one allocator it does not expose, or a serving
// loop that must never call cudaMalloc because that call can synchronise the
// whole device and stall the other streams.  h3dit_block_forward_noalloc
// serves them with a fixed scratch area that lives in the library's own
// device image, so neither the caller nor the library allocates anything.
namespace {

// 64 MiB of block workspace (the tiny-block class and other small shapes fit;
// a full-width block at thousands of tokens does not and is refused).  Every
// GPU that loads the library holds this array until the process exits.
constexpr size_t kStaticScratchBytes = size_t(64) << 20;
static __device__ __align__(256) uint8_t g_static_scratch[kStaticScratchBytes];

std::mutex g_static_mu;
void* g_static_addr[64] = {nullptr};

// Device address of g_static_scratch on the current device, looked up once
// per device (the first call on that device) and kept for the life of the
// process.  On the host the array's name only stands in for the symbol;
// passing it to a kernel would be wrong, so the real address comes from the
// runtime.  cudaDeviceReset unloads the module, so the kept address is not
// valid after one: the header says a reset ends the use of this entry point.
h3dit_status static_scratch_address(void** out) {
  int dev = -1;
  H3_CUDA(cudaGetDevice(&dev));
  if (dev < 0 || dev >= 64) return fail(H3DIT_E_UNSUPPORTED, "device ordinal %d out of range", dev);
  std::lock_guard<std::mutex> lk(g_static_mu);
  if (!g_static_addr[dev]) {
    void* p = nullptr;
    H3_CUDA(cudaGetSymbolAddress(&p, g_static_scratch));
    if (!p || !aligned(p, 256)) return fail(H3DIT_E_CUDA, "static scratch address is not usable");
    g_static_addr[dev] = p;
  }
  *out = g_static_addr[dev];
  return H3DIT_OK;
}

}  // namespace

extern "C" h3dit_status h3dit_block_forward_noalloc(const h3dit_config* cfg, const h3dit_block_weights* w,
                                                    const float* mod, void* x, const float* pos, int n_tokens,
                                                    cudaStream_t stream) {
  // the same argument checks as h3dit_block_forward, in the same order,
  // before the size of the built-in scratch is considered
  H3_TRY(check_cfg(cfg));
  H3_TRY(check_weights(cfg, w));
  if (!mod || !x || !pos) return fail(H3DIT_E_INVAL, "NULL pointer");
  if (n_tokens < 1) return fail(H3DIT_E_INVAL, "n_tokens %d", n_tokens);
  if (!aligned(x, 16)) return fail(H3DIT_E_INVAL, "x must be 16-byte aligned");
  const size_t need = plan_arena(cfg, n_tokens, nullptr).total;
  if (need > kStaticScratchBytes)
    return fail(H3DIT_E_NOMEM,
                "block at %d tokens needs %zu bytes of scratch; the built-in scratch holds %zu bytes "
                "(use h3dit_block_forward with a caller workspace)",
                n_tokens, need, kStaticScratchBytes);
  void* ws = nullptr;
  H3_TRY(static_scratch_address(&ws));
  // Nothing in the scratch has to start at zero: every byte the block reads
  // from it is written earlier in the same call.
  return h3dit_block_forward(cfg, w, mod, x, pos, n_tokens, ws, kStaticScratchBytes, stream);
}
