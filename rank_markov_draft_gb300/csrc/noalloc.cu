// noalloc.cu -- dspark_markov_draft_noalloc: the vanilla Markov-head draft
// without a context and without any device allocation.
//
// Who needs this: callers that are not allowed to allocate device memory on
// their own, such as a library embedded in a host framework that owns every
// byte of device memory through its own pool (a stray cudaMalloc would bypass
// the pool's accounting and fragment it), or a serving loop that forbids
// cudaMalloc / cudaFree on its hot path because they can synchronise the
// device.  Such callers still pass their own inputs and outputs.
//
// How: the draft kernel's scratch (grid-barrier counter, status word,
// per-step argmax keys and cross-CTA partials) lives in one file-scope
// __device__ array of a fixed size, loaded with the library on every GPU and
// kept until the process exits.  Host code cannot use the array's name as a
// device address (on the host it is only a stand-in symbol), so its device
// address is looked up with cudaGetSymbolAddress while the device is current,
// and passed to the kernel.  The look-up is done once per CUDA context: the
// cache is keyed on the current context's process-unique id (cuCtxGetId), so a
// context created after cudaDeviceReset (which reloads the module and can
// move the array) gets a fresh look-up instead of a stale address.
//
// The array is shared by every call on a device and keeps the contents of the
// last call: each call clears the counter, status and keys on its stream
// before launching.  Calls whose work overlaps on the GPU (different streams,
// or other host threads) race on the array; callers must serialise them.

#include <cstring>
#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>

#include "dspark.h"
#include "internal.h"
#include "philox.cuh"

namespace {

// Limits of the context-free entry point.
constexpr int kNaMaxK = 16;       // block positions
constexpr int kNaMaxGrid = 160;   // CTAs (one per SM; GB300 has 152)
constexpr int kNaMaxDevices = 64;
// key epochs of the draft kernel are 14-bit (1 .. 16383): one per 128-request chunk
constexpr int kNaMaxChunks = 16383;
constexpr int kNaMaxBatch = kNaMaxChunks * dspark::kBatchChunk;

constexpr size_t kNaOffBar = 0;         // uint32_t grid-barrier counter
constexpr size_t kNaOffStatus = 4;      // int device status
constexpr size_t kNaOffKeys = 256;      // uint64_t [kNaMaxK][128]
constexpr size_t kNaKeysBytes = sizeof(unsigned long long) * kNaMaxK * dspark::kBatchChunk;
constexpr size_t kNaOffPartials = kNaOffKeys + kNaKeysBytes;
constexpr size_t kNaPartialsBytes =
    sizeof(dspark::DraftPartial) * kNaMaxK * dspark::kBatchChunk * kNaMaxGrid;
constexpr size_t kNaScratchBytes = kNaOffPartials + kNaPartialsBytes;  // ~7.9 MB

static_assert(kNaOffPartials % 256 == 0, "partials must stay 256-byte aligned");

// The scratch itself: a fixed-size, 256-byte aligned device array.
static __device__ __align__(256) unsigned char g_draft_scratch[kNaScratchBytes];

std::mutex g_setup_mutex;
// device address of g_draft_scratch per device, valid for the context it was looked up in
void* g_scratch_ptr[kNaMaxDevices] = {};
unsigned long long g_scratch_ctx[kNaMaxDevices] = {};  // that context's id (0: none yet)

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

bool encode(CUtensorMap* map, CUtensorMapDataType dt, const void* base, int rank,
            const cuuint64_t* dims, const cuuint64_t* strides, const cuuint32_t* box) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint32_t elem[4] = {1, 1, 1, 1};  // rank <= 4
  return fn(map, dt, rank, const_cast<void*>(base), dims, strides, box, elem,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

// Process-unique id of the calling thread's current CUDA context (0 on failure).
unsigned long long current_context_id() {
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<CtxGetCurrentFn>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetIdFn>(p);
  });
  if (get_current == nullptr || get_id == nullptr) return 0;
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return 0;
  if (get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

// Set-up on the current device, once per CUDA context: the scratch's device address.
// If no context is current yet on this thread, cudaGetSymbolAddress initialises the
// device's primary context (and makes it current) before the id is read.
int scratch_for_current_device(int device, unsigned char** out) {
  if (device < 0 || device >= kNaMaxDevices) return DSPARK_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  unsigned long long ctx_id = current_context_id();  // 0: no context current yet
  if (ctx_id == 0 || g_scratch_ptr[device] == nullptr || g_scratch_ctx[device] != ctx_id) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_draft_scratch) != cudaSuccess || ptr == nullptr)
      return DSPARK_ERR_CUDA;
    ctx_id = current_context_id();
    if (ctx_id == 0) return DSPARK_ERR_CUDA;
    g_scratch_ptr[device] = ptr;
    g_scratch_ctx[device] = ctx_id;
  }
  *out = static_cast<unsigned char*>(g_scratch_ptr[device]);
  return DSPARK_OK;
}

}  // namespace

extern "C" int dspark_markov_draft_noalloc(const float* U, const uint16_t* W1, const uint16_t* W2,
                                           const int32_t* anchors, int B, int K, int V, int r,
                                           float temperature, uint64_t seed, int32_t* tokens,
                                           float* logprobs, int* device_status,
                                           dspark_stream_t stream) {
  // argument checks (nothing is enqueued on failure)
  if (U == nullptr || anchors == nullptr || tokens == nullptr || logprobs == nullptr)
    return DSPARK_ERR_INVALID_ARG;
  if (B <= 0 || K <= 0 || V <= 0) return DSPARK_ERR_INVALID_ARG;
  if (K > kNaMaxK) return DSPARK_ERR_CAPACITY;  // the fixed scratch holds 16 positions
  if (B > kNaMaxBatch) return DSPARK_ERR_CAPACITY;  // one 14-bit key epoch per 128 requests
  if (V > (1 << 18) || (V % 8) != 0) return DSPARK_ERR_UNSUPPORTED;
  if (r < 0) return DSPARK_ERR_INVALID_ARG;
  if (r > dspark::kMaxRank || (r % 16) != 0) return DSPARK_ERR_UNSUPPORTED;
  if (r > 0 && (W1 == nullptr || W2 == nullptr)) return DSPARK_ERR_INVALID_ARG;
  if (!(temperature >= 0.f) || temperature > 3.0e38f) return DSPARK_ERR_INVALID_ARG;
  if (!aligned16(U) || !aligned16(anchors) || (W1 && !aligned16(W1)) || (W2 && !aligned16(W2)))
    return DSPARK_ERR_INVALID_ARG;

  int device = 0;
  if (cudaGetDevice(&device) != cudaSuccess) return DSPARK_ERR_NO_DEVICE;
  int major = 0, minor = 0, sms = 0, coop = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, device) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, device) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess ||
      cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, device) != cudaSuccess)
    return DSPARK_ERR_CUDA;
  if (major != 10 || minor != 3 || !coop) return DSPARK_ERR_NO_DEVICE;
  unsigned char* scratch = nullptr;
  int st = scratch_for_current_device(device, &scratch);
  if (st != DSPARK_OK) return st;

  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  uint32_t* bar = reinterpret_cast<uint32_t*>(scratch + kNaOffBar);
  int* status = reinterpret_cast<int*>(scratch + kNaOffStatus);
  unsigned long long* keys = reinterpret_cast<unsigned long long*>(scratch + kNaOffKeys);
  dspark::DraftPartial* partials = reinterpret_cast<dspark::DraftPartial*>(scratch + kNaOffPartials);
  // the array keeps the previous call's contents: clear what must start at zero
  if (cudaMemsetAsync(scratch, 0, kNaOffPartials, s) != cudaSuccess) return DSPARK_ERR_CUDA;

  const int n_tiles = (V + dspark::kDraftTileN - 1) / dspark::kDraftTileN;
  int grid = n_tiles < sms ? n_tiles : sms;
  if (grid > kNaMaxGrid) grid = kNaMaxGrid;
  const float inv_t = temperature > 0.f ? 1.0f / temperature : 1.0f;
  const int mode = temperature > 0.f ? dspark::kModeSample : dspark::kModeGreedy;
  uint32_t bar_base = 0, epoch = 0;
  for (int b0 = 0; b0 < B; b0 += dspark::kBatchChunk) {
    const int Bc = (B - b0) < dspark::kBatchChunk ? (B - b0) : dspark::kBatchChunk;
    dspark::DraftArgs args;
    std::memset(&args, 0, sizeof(args));
    if (r > 0) {
      const cuuint64_t dims[2] = {static_cast<cuuint64_t>(V), static_cast<cuuint64_t>(r)};
      const cuuint64_t strides[1] = {static_cast<cuuint64_t>(V) * 2};
      const cuuint32_t box[2] = {static_cast<cuuint32_t>(dspark::kDraftBoxV),
                                 static_cast<cuuint32_t>(dspark::draft_slice_rows(r))};
      if (!encode(&args.tm_w2, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, W2, 2, dims, strides, box))
        return DSPARK_ERR_CUDA;
    }
    const int box_rows = (Bc + 7) & ~7;
    // U boxes of row pairs (256 contiguous bytes a row) above 64 requests
    const bool rowpair = V % 32 == 0 && Bc > 64;
    if (rowpair) {
      const cuuint64_t dims[4] = {32, static_cast<cuuint64_t>(V) / 32,
                                  static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(Bc)};
      const cuuint64_t strides[3] = {128, static_cast<cuuint64_t>(V) * 4,
                                     static_cast<cuuint64_t>(K) * V * 4};
      const cuuint32_t box[4] = {32, 2, 1,
                                 static_cast<cuuint32_t>(box_rows > 64 ? 64 : box_rows)};
      if (!encode(&args.tm_u, CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
                  U + static_cast<size_t>(b0) * K * V, 4, dims, strides, box))
        return DSPARK_ERR_CUDA;
    } else {
      const cuuint64_t dims[3] = {static_cast<cuuint64_t>(V), static_cast<cuuint64_t>(K),
                                  static_cast<cuuint64_t>(Bc)};
      const cuuint64_t strides[2] = {static_cast<cuuint64_t>(V) * 4,
                                     static_cast<cuuint64_t>(K) * V * 4};
      const cuuint32_t box[3] = {32, 1, static_cast<cuuint32_t>(box_rows)};
      if (!encode(&args.tm_u, CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
                  U + static_cast<size_t>(b0) * K * V, 3, dims, strides, box))
        return DSPARK_ERR_CUDA;
    }
    dspark::DraftParams& p = args.p;
    p.W1 = W1;
    p.anchors = anchors + b0;
    p.B = Bc;
    p.K = K;
    p.V = V;
    p.r = r;
    p.b_global0 = b0;
    p.n_tiles = n_tiles;
    p.box_rows = box_rows;
    p.u_rowpair = rowpair ? 1 : 0;
    p.inv_t = inv_t;
    p.seed_lo = static_cast<uint32_t>(seed & 0xFFFFFFFFull);
    p.seed_hi = static_cast<uint32_t>(seed >> 32);
    dspark::philox_round_keys(p.seed_lo, p.seed_hi, p.round_key0, p.round_key1);
    p.tokens = tokens + static_cast<size_t>(b0) * K;
    p.logprobs = logprobs + static_cast<size_t>(b0) * K;
    p.keys = keys;
    p.partials = partials;
    p.bar = bar;
    p.status = status;
    p.bar_base = bar_base;
    p.epoch = ++epoch;  // keys were cleared at the start of this call
    p.debug_skip_cta = -1;
    p.timeout_ns = dspark::kDefaultTimeoutNs;
    if (dspark::launch_draft(args, mode, grid, s) != cudaSuccess) return DSPARK_ERR_CUDA;
    bar_base += static_cast<uint32_t>(K) * static_cast<uint32_t>(grid);
  }
  if (device_status != nullptr &&
      cudaMemcpyAsync(device_status, status, sizeof(int), cudaMemcpyDeviceToDevice, s) !=
          cudaSuccess)
    return DSPARK_ERR_CUDA;
  return DSPARK_OK;
}
