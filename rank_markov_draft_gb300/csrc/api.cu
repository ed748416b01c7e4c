// api.cu -- the C ABI declared in include/dspark.h: argument validation,
// context scratch, TMA tensor-map encoding and kernel dispatch.  Every step of
// the hot path runs in this library's kernels; the host code only checks,
// describes and enqueues.

#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>

#include "dspark.h"
#include "internal.h"
#include "philox.cuh"

using dspark::DraftArgs;
using dspark::DraftParams;
using dspark::DraftPartial;
using dspark::GateArgs;

struct dspark_ctx {
  int device = 0;
  int num_sms = 0;
  int B_max = 0, V_max = 0, K_max = 0;
  int* d_status = nullptr;
  uint32_t* d_bar = nullptr;
  unsigned long long* d_keys = nullptr;  // [K_max][128]
  DraftPartial* d_partials = nullptr;    // [K_max][128][num_sms]
  float* d_H = nullptr;                  // [B_max * K_max][256] gate, fp32 (pair scores, preps)
  uint16_t* d_Hb = nullptr;              // the gate in bf16 for the draft kernel (RNN: input gate)
  uint16_t* d_Ab = nullptr;              // [B_max * K_max][256] bf16 decay gate of the RNN head
  float* d_gate_part = nullptr;          // [kGateSplitsMax][B_max * K_max][256]
  int32_t* d_topk_part_i = nullptr;      // [kTopkPartUnits][kMaxTopk] per-piece top-k lists
  // verification scratch
  float* d_v_lse_t = nullptr;            // [B_max][K_max + 1]
  int32_t* d_v_argmax_t = nullptr;       // [B_max][K_max + 1]
  uint16_t* d_v_H = nullptr;             // [B_max][256] bf16
  int32_t* d_v_prev = nullptr;           // [B_max]
  dspark::ResRow* d_v_rows = nullptr;    // [B_max]
  // verification's per-request scratch, zero between calls
  unsigned long long* d_v_fail = nullptr;  // [B_max]
  int* d_v_count = nullptr;                // [B_max]
  // acceptance-label scratch
  int32_t* d_l_prev = nullptr;           // [B_max * K_max] predecessors of the drafted tokens
  float* d_l_offq2 = nullptr;            // [B_max * K_max] log2 q offsets
  float* d_topk_part_v = nullptr;
  uint32_t bar_counter = 0;              // host copy of the grid-barrier counter
  uint32_t epoch = 0;                    // last key epoch used
  int poisoned = 0;
  int debug_skip_cta = -1;
  bool debug_refuse_launch = false;  // the next draft launch asks for too much shared memory
  uint64_t timeout_ns = dspark::kDefaultTimeoutNs;
  int last_launches = 0;
  unsigned long long* trace = nullptr;  // caller's device buffer for the next draft's phase trace
  int64_t trace_capacity = 0;
};

namespace {

constexpr int kGateSplitsMax = 8;
constexpr uint32_t kEpochMax = 16383;

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
        q == cudaDriverEntryPointSuccess) {
      fn = reinterpret_cast<EncodeTiledFn>(p);
    }
  });
  return fn;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool encode_2d(CUtensorMap* map, CUtensorMapDataType dt, const void* base, uint64_t inner,
               uint64_t outer, uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t elem[2] = {1, 1};
  return fn(map, dt, 2, const_cast<void*>(base), dims, strides, box, elem,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// A [Bc][K][V] fp32 array (U, or the target's [Bc][K + 1][V]) as [Bc][K][V / 32][32]
// (V % 32 == 0), boxes of 2 chunks x min(box_rows, 64) rows: each box reads 256 contiguous
// bytes of every row it holds
bool encode_u_rowpair(CUtensorMap* map, const float* base, int V, int K, int Bc, int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[4] = {32, static_cast<cuuint64_t>(V) / 32, static_cast<cuuint64_t>(K),
                              static_cast<cuuint64_t>(Bc)};
  const cuuint64_t strides[3] = {128, static_cast<cuuint64_t>(V) * 4,
                                 static_cast<cuuint64_t>(K) * V * 4};
  const cuuint32_t box[4] = {32, 2, 1, static_cast<cuuint32_t>(box_rows > 64 ? 64 : box_rows)};
  const cuuint32_t elem[4] = {1, 1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, const_cast<float*>(base), dims, strides, box,
            elem, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_3d(CUtensorMap* map, CUtensorMapDataType dt, const void* base, uint64_t d0,
               uint64_t d1, uint64_t d2, uint64_t s1, uint64_t s2, uint32_t b0, uint32_t b1,
               uint32_t b2, CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[3] = {d0, d1, d2};
  const cuuint64_t strides[2] = {s1, s2};
  const cuuint32_t box[3] = {b0, b1, b2};
  const cuuint32_t elem[3] = {1, 1, 1};
  return fn(map, dt, 3, const_cast<void*>(base), dims, strides, box, elem,
            CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int check_rank(int r) {
  if (r < 0) return DSPARK_ERR_INVALID_ARG;
  if (r > dspark::kMaxRank || (r % 16) != 0) return DSPARK_ERR_UNSUPPORTED;
  return DSPARK_OK;
}

int check_conf(const dspark_conf_args* conf, int r) {
  if (conf == nullptr) return DSPARK_OK;
  if (conf->h == nullptr || conf->w == nullptr || conf->conf == nullptr ||
      conf->cumprod == nullptr || conf->verify_len == nullptr)
    return DSPARK_ERR_INVALID_ARG;
  if (conf->d <= 0 || (conf->d % 8) != 0) return DSPARK_ERR_INVALID_ARG;
  // the Markov embedding needs a Markov head (vLLM guide: rank 0 pairs with
  // --no-confidence-head-with-markov)
  if (conf->with_markov && r == 0) return DSPARK_ERR_INVALID_ARG;
  if (!aligned16(conf->h) || !aligned16(conf->w)) return DSPARK_ERR_INVALID_ARG;
  if (!(conf->threshold == conf->threshold)) return DSPARK_ERR_INVALID_ARG;
  return DSPARK_OK;
}

int check_ctx(dspark_ctx* ctx) {
  if (ctx == nullptr) return DSPARK_ERR_INVALID_ARG;
  if (ctx->poisoned) return DSPARK_ERR_CTX_POISONED;
  if (cudaSetDevice(ctx->device) != cudaSuccess) return DSPARK_ERR_CUDA;
  return DSPARK_OK;
}

int cuda_status(cudaError_t e) { return e == cudaSuccess ? DSPARK_OK : DSPARK_ERR_CUDA; }

// Next key epoch; keys of older epochs always lose an atomicMax against it.
int next_epoch(dspark_ctx* ctx, cudaStream_t stream, uint32_t* epoch) {
  if (ctx->epoch >= kEpochMax) {
    if (cudaMemsetAsync(ctx->d_keys, 0,
                        sizeof(unsigned long long) * ctx->K_max * dspark::kBatchChunk,
                        stream) != cudaSuccess)
      return DSPARK_ERR_CUDA;
    ctx->epoch = 0;
  }
  *epoch = ++ctx->epoch;
  return DSPARK_OK;
}

// Gate prologue into H [M, r] fp32 and/or Hb [M, r] bf16 (either may be null; they may be
// the context's buffers).
int run_gate(dspark_ctx* ctx, const uint16_t* h, const uint16_t* Wg, int M, int d, int r,
             float* H, uint16_t* Hb, cudaStream_t stream) {
  GateArgs ga{};
  if (!encode_2d(&ga.tm_h, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, h, d, M, static_cast<uint64_t>(d) * 2,
                 64, 128))
    return DSPARK_ERR_CUDA;
  if (!encode_2d(&ga.tm_wg, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, Wg, r, d,
                 static_cast<uint64_t>(r) * 2, 64, 64))
    return DSPARK_ERR_CUDA;
  const int nchunks = d / 64;
  const int base = ((M + 127) / 128) * (r / 64);
  int splits = ctx->num_sms / (base > 0 ? base : 1);
  if (splits < 1) splits = 1;
  if (splits > kGateSplitsMax) splits = kGateSplitsMax;
  if (splits > nchunks) splits = nchunks;
  const int cps = (nchunks + splits - 1) / splits;
  splits = (nchunks + cps - 1) / cps;  // every split gets at least one chunk
  ga.partial = ctx->d_gate_part;
  ga.M = M;
  ga.d = d;
  ga.r = r;
  ga.splits = splits;
  ga.chunks_per_split = cps;
  ga.status = ctx->d_status;
  ga.timeout_ns = ctx->timeout_ns;
  cudaError_t e = dspark::launch_gate_gemm(ga, stream);
  if (e != cudaSuccess) return DSPARK_ERR_CUDA;
  e = dspark::launch_gate_finalize(ctx->d_gate_part, splits, static_cast<int64_t>(M) * r, H, Hb,
                                   stream);
  ctx->last_launches += 2;
  return cuda_status(e);
}

// Inputs of the draft kernel's acceptance-label mode (whole call; chunked below).
struct LabelIn {
  const float* target;  // [B, K+1, V] target logits (label; residual: with K = res_K)
  const float* lse_t;   // [B, K+1] (label)
  const float* offq2;   // [B, K] (label)
  float* label;         // [B, K] (label)
  float target_scale2;  // log2(e) / Tt
  const dspark::ResRow* rows;  // [B] (residual), else null
  int res_K;            // residual: K of the caller's U [B, K, V] (passed as U) and target
};

// The persistent draft kernel over chunks of 128 requests.
int run_draft(dspark_ctx* ctx, int mode, const float* U, const uint16_t* W1, const uint16_t* W2,
              const int32_t* anchors, const int32_t* prev, const uint16_t* H, int B, int K, int V,
              int r, float temperature, uint64_t seed, int32_t* tokens, float* logprobs,
              float* logits, float* lse, const dspark_conf_args* conf, cudaStream_t stream,
              const LabelIn* lab = nullptr, const uint16_t* Agate = nullptr) {
  const int n_tiles = (V + dspark::kDraftTileN - 1) / dspark::kDraftTileN;
  const int grid = n_tiles < ctx->num_sms ? n_tiles : ctx->num_sms;
  const float inv_t = temperature > 0.f ? 1.0f / temperature : 1.0f;
  for (int b0 = 0; b0 < B; b0 += dspark::kBatchChunk) {
    const int Bc = (B - b0) < dspark::kBatchChunk ? (B - b0) : dspark::kBatchChunk;
    DraftArgs args;
    std::memset(&args, 0, sizeof(args));
    if (r > 0 && !encode_2d(&args.tm_w2, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, W2, V, r,
                            static_cast<uint64_t>(V) * 2, dspark::kDraftBoxV,
                            dspark::draft_slice_rows(r)))
      return DSPARK_ERR_CUDA;
    const int box_rows = (Bc + 7) & ~7;
    const bool res = lab != nullptr && lab->rows != nullptr;
    // row-pair U boxes (256 contiguous bytes a row and box, against 128 for 32-token boxes:
    // the U stream reaches about 6.3 TB/s instead of 4.5) where V allows them: for the label
    // pass, and for the modes that read U alone above 64 requests (at 64 or fewer the batch
    // copies' 32-token boxes measured faster); not for the residual draw's gathered rows
    const bool rowpair = V % 32 == 0 && (lab != nullptr ? !res : Bc > 64);
    if (res) {
      // the draw rows are gathered in place: U and the target as plain row arrays
      const uint64_t Kr = static_cast<uint64_t>(lab->res_K);
      if (!encode_2d(&args.tm_u, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, U, V, B * Kr,
                     static_cast<uint64_t>(V) * 4, 32, 1) ||
          !encode_2d(&args.tm_p, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, lab->target, V, B * (Kr + 1),
                     static_cast<uint64_t>(V) * 4, 32, 1))
        return DSPARK_ERR_CUDA;
    } else if (rowpair) {
      // (the label pass's fills take rows [0, 64) and [64, 128) in turn: 64-row boxes)
      if (!encode_u_rowpair(&args.tm_u, U + static_cast<size_t>(b0) * K * V, V, K, Bc,
                            lab != nullptr ? 64 : box_rows))
        return DSPARK_ERR_CUDA;
    } else {
      const float* Uc = U + static_cast<size_t>(b0) * K * V;
      if (!encode_3d(&args.tm_u, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, Uc, V, K, Bc,
                     static_cast<uint64_t>(V) * 4, static_cast<uint64_t>(K) * V * 4, 32, 1,
                     box_rows))
        return DSPARK_ERR_CUDA;
    }
    DraftParams& p = args.p;
    p.W1 = W1;
    p.anchors = anchors + b0;
    p.prev = prev ? prev + static_cast<size_t>(b0) * K : nullptr;
    p.H = H ? H + static_cast<size_t>(b0) * K * r : nullptr;
    p.A = Agate ? Agate + static_cast<size_t>(b0) * K * r : nullptr;
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
    const size_t o = static_cast<size_t>(b0) * K;
    p.tokens = tokens ? tokens + o : nullptr;
    p.logprobs = logprobs ? logprobs + o : nullptr;
    p.logits = logits ? logits + o * V : nullptr;
    p.lse = lse ? lse + o : nullptr;
    if (lab != nullptr) {
      p.target_scale2 = lab->target_scale2;
      if (res) {
        p.rows = lab->rows + b0;
        p.res_K = lab->res_K;
      } else {
        const float* tchunk = lab->target + static_cast<size_t>(b0) * (K + 1) * V;
        if (rowpair ? !encode_u_rowpair(&args.tm_p, tchunk, V, K + 1, Bc, 64)
                    : !encode_3d(&args.tm_p, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, tchunk, V, K + 1,
                                 Bc, static_cast<uint64_t>(V) * 4,
                                 static_cast<uint64_t>(K + 1) * V * 4, 32, 1, box_rows))
          return DSPARK_ERR_CUDA;
        p.target = tchunk;
        p.lse_t = lab->lse_t + static_cast<size_t>(b0) * (K + 1);
        p.offq2 = lab->offq2 + o;
        p.label = lab->label + o;
      }
    }
    if (conf != nullptr) {
      p.conf_h = conf->h + o * conf->d;
      p.conf_w = conf->w;
      p.conf_bias = conf->bias;
      p.conf_d = conf->d;
      p.conf_with_markov = conf->with_markov;
      p.conf_threshold = conf->threshold;
      p.conf_tau = conf->tau;
      p.conf = conf->conf + o;
      p.cumprod = conf->cumprod + o;
      p.verify_len = conf->verify_len + b0;
    }
    p.keys = ctx->d_keys;
    p.partials = ctx->d_partials;
    p.bar = ctx->d_bar;
    p.status = ctx->d_status;
    p.bar_base = ctx->bar_counter;
    int st = next_epoch(ctx, stream, &p.epoch);
    if (st != DSPARK_OK) return st;
    p.debug_skip_cta = ctx->debug_skip_cta;
    p.timeout_ns = ctx->timeout_ns;
    if (ctx->trace != nullptr &&
        static_cast<int64_t>(grid) * K * dspark::kTraceSlots <= ctx->trace_capacity && b0 == 0)
      p.trace = ctx->trace;
    const uint32_t extra = ctx->debug_refuse_launch ? 1024u : 0u;
    ctx->debug_refuse_launch = false;
    // the first chunk of a call that has just run its own kernel (the label and residual
    // passes after the scan that writes their per-row inputs, the gated and RNN heads after
    // their gate GEMMs) is launched as that kernel's programmatic dependent (not after a key
    // reset, whose memset would then be the preceding work)
    const bool dependent = (lab != nullptr || H != nullptr) && b0 == 0 && p.epoch != 1;
    cudaError_t e = dspark::launch_draft(args, mode, grid, stream, extra, dependent);
    if (e != cudaSuccess) {
      ctx->debug_skip_cta = -1;
      ctx->trace = nullptr;
      return DSPARK_ERR_CUDA;
    }
    ctx->bar_counter += static_cast<uint32_t>(K) * static_cast<uint32_t>(grid);
    ctx->last_launches += 1;
  }
  ctx->debug_skip_cta = -1;  // the fault-injection and trace knobs cover one call
  ctx->trace = nullptr;
  return DSPARK_OK;
}

int check_draft_args(const float* U, const uint16_t* W1, const uint16_t* W2,
                     const int32_t* anchors, int B, int K, int V, int r, float temperature,
                     const void* out0, const void* out1) {
  if (U == nullptr || anchors == nullptr || out0 == nullptr || out1 == nullptr)
    return DSPARK_ERR_INVALID_ARG;
  if (B <= 0 || K <= 0 || V <= 0) return DSPARK_ERR_INVALID_ARG;
  if (K > dspark::kMaxK || V > (1 << 18)) return DSPARK_ERR_UNSUPPORTED;
  if ((V % 8) != 0) return DSPARK_ERR_UNSUPPORTED;
  const int rs = check_rank(r);
  if (rs != DSPARK_OK) return rs;
  if (r > 0 && (W1 == nullptr || W2 == nullptr)) return DSPARK_ERR_INVALID_ARG;
  if (!(temperature >= 0.f) || temperature > 3.0e38f) return DSPARK_ERR_INVALID_ARG;
  if (!aligned16(U) || !aligned16(anchors) || (W1 && !aligned16(W1)) || (W2 && !aligned16(W2)))
    return DSPARK_ERR_INVALID_ARG;
  return DSPARK_OK;
}

int check_gate_args(const uint16_t* h, const uint16_t* Wg, int d, int r) {
  if (h == nullptr || Wg == nullptr) return DSPARK_ERR_INVALID_ARG;
  if (d <= 0) return DSPARK_ERR_INVALID_ARG;
  if ((d % 64) != 0 || r <= 0 || (r % 64) != 0 || r > dspark::kMaxRank)
    return DSPARK_ERR_UNSUPPORTED;
  if (!aligned16(h) || !aligned16(Wg)) return DSPARK_ERR_INVALID_ARG;
  return DSPARK_OK;
}

// Gates of the RNN head into the context, in bf16: decay a = sigmoid(h . Wa) into d_Ab, and
// the input gate g = sigmoid(h . Wg) into d_Hb when Wg is given (else g = 1: H stays null).
int run_rnn_gates(dspark_ctx* ctx, const uint16_t* h, const uint16_t* Wa, const uint16_t* Wg,
                  int M, int d, int r, const uint16_t** H, cudaStream_t s) {
  int st = run_gate(ctx, h, Wa, M, d, r, nullptr, ctx->d_Ab, s);
  if (st != DSPARK_OK) return st;
  *H = nullptr;
  if (Wg != nullptr) {
    st = run_gate(ctx, h, Wg, M, d, r, nullptr, ctx->d_Hb, s);
    if (st != DSPARK_OK) return st;
    *H = ctx->d_Hb;
  }
  return DSPARK_OK;
}

int check_rnn_args(const uint16_t* h, const uint16_t* Wa, const uint16_t* Wg, int d, int r) {
  int st = check_gate_args(h, Wa, d, r);
  if (st != DSPARK_OK) return st;
  if (Wg != nullptr && (st = check_gate_args(h, Wg, d, r)) != DSPARK_OK) return st;
  return DSPARK_OK;
}

}  // namespace

extern "C" {

const char* dspark_strerror(int code) {
  switch (code) {
    case DSPARK_OK: return "ok";
    case DSPARK_ERR_INVALID_ARG: return "invalid argument";
    case DSPARK_ERR_UNSUPPORTED: return "unsupported shape or option";
    case DSPARK_ERR_CUDA: return "CUDA call failed";
    case DSPARK_ERR_TIMEOUT: return "device wait timed out (kernel exited cleanly)";
    case DSPARK_ERR_DEVICE_OOB: return "token id out of range on the device";
    case DSPARK_ERR_NO_DEVICE: return "no usable sm_103 device";
    case DSPARK_ERR_CTX_POISONED: return "context poisoned by an earlier device error";
    case DSPARK_ERR_CAPACITY: return "size above the context's creation limits";
    default: return "unknown status";
  }
}

int dspark_abi_version(void) { return DSPARK_ABI_VERSION; }

int dspark_ctx_create(dspark_ctx** out, int device, int B_max, int V_max, int K_max) {
  if (out == nullptr) return DSPARK_ERR_INVALID_ARG;
  *out = nullptr;
  if (B_max <= 0 || V_max <= 0 || K_max <= 0) return DSPARK_ERR_INVALID_ARG;
  if (K_max > dspark::kMaxK || V_max > (1 << 18)) return DSPARK_ERR_UNSUPPORTED;
  int ndev = 0;
  if (cudaGetDeviceCount(&ndev) != cudaSuccess || device < 0 || device >= ndev)
    return DSPARK_ERR_NO_DEVICE;
  cudaDeviceProp prop{};
  if (cudaGetDeviceProperties(&prop, device) != cudaSuccess) return DSPARK_ERR_CUDA;
  if (prop.major != 10 || prop.minor != 3) return DSPARK_ERR_NO_DEVICE;
  if (!prop.cooperativeLaunch) return DSPARK_ERR_NO_DEVICE;
  if (cudaSetDevice(device) != cudaSuccess) return DSPARK_ERR_CUDA;
  if (encode_fn() == nullptr) return DSPARK_ERR_CUDA;
  dspark_ctx* ctx = new dspark_ctx();
  ctx->device = device;
  ctx->num_sms = prop.multiProcessorCount;
  ctx->B_max = B_max;
  ctx->V_max = V_max;
  ctx->K_max = K_max;
  const size_t rows = static_cast<size_t>(B_max) * K_max;
  bool ok = cudaMalloc(&ctx->d_status, sizeof(int)) == cudaSuccess &&
            cudaMalloc(&ctx->d_bar, sizeof(uint32_t)) == cudaSuccess &&
            cudaMalloc(&ctx->d_keys, sizeof(unsigned long long) * K_max * dspark::kBatchChunk) ==
                cudaSuccess &&
            cudaMalloc(&ctx->d_partials, sizeof(DraftPartial) * static_cast<size_t>(K_max) *
                                             dspark::kBatchChunk * ctx->num_sms) == cudaSuccess &&
            cudaMalloc(&ctx->d_H, sizeof(float) * rows * dspark::kMaxRank) == cudaSuccess &&
            cudaMalloc(&ctx->d_Hb, sizeof(uint16_t) * rows * dspark::kMaxRank) == cudaSuccess &&
            cudaMalloc(&ctx->d_Ab, sizeof(uint16_t) * rows * dspark::kMaxRank) == cudaSuccess &&
            cudaMalloc(&ctx->d_gate_part,
                       sizeof(float) * kGateSplitsMax * rows * dspark::kMaxRank) == cudaSuccess &&
            cudaMalloc(&ctx->d_topk_part_i, sizeof(int32_t) * dspark::kTopkPartUnits *
                                                dspark::kMaxTopk) == cudaSuccess &&
            cudaMalloc(&ctx->d_topk_part_v,
                       sizeof(float) * dspark::kTopkPartUnits * dspark::kMaxTopk) == cudaSuccess &&
            cudaMalloc(&ctx->d_v_lse_t, sizeof(float) * B_max * (K_max + 1)) == cudaSuccess &&
            cudaMalloc(&ctx->d_v_argmax_t, sizeof(int32_t) * B_max * (K_max + 1)) == cudaSuccess &&
            cudaMalloc(&ctx->d_v_H, sizeof(uint16_t) * B_max * dspark::kMaxRank) == cudaSuccess &&
            cudaMalloc(&ctx->d_v_prev, sizeof(int32_t) * B_max) == cudaSuccess &&
            cudaMalloc(&ctx->d_v_rows, sizeof(dspark::ResRow) * B_max) == cudaSuccess &&
            cudaMalloc(&ctx->d_v_fail, sizeof(unsigned long long) * B_max) == cudaSuccess &&
            cudaMalloc(&ctx->d_v_count, sizeof(int) * B_max) == cudaSuccess &&
            cudaMalloc(&ctx->d_l_prev, sizeof(int32_t) * rows) == cudaSuccess &&
            cudaMalloc(&ctx->d_l_offq2, sizeof(float) * rows) == cudaSuccess;
  ok = ok && cudaMemset(ctx->d_status, 0, sizeof(int)) == cudaSuccess &&
       cudaMemset(ctx->d_bar, 0, sizeof(uint32_t)) == cudaSuccess &&
       cudaMemset(ctx->d_keys, 0, sizeof(unsigned long long) * K_max * dspark::kBatchChunk) ==
           cudaSuccess &&
       cudaMemset(ctx->d_v_fail, 0, sizeof(unsigned long long) * B_max) == cudaSuccess &&
       cudaMemset(ctx->d_v_count, 0, sizeof(int) * B_max) == cudaSuccess &&
       cudaDeviceSynchronize() == cudaSuccess;
  if (!ok) {
    dspark_ctx_destroy(ctx);
    return DSPARK_ERR_CUDA;
  }
  *out = ctx;
  return DSPARK_OK;
}

int dspark_ctx_destroy(dspark_ctx* ctx) {
  if (ctx == nullptr) return DSPARK_ERR_INVALID_ARG;
  cudaSetDevice(ctx->device);
  cudaFree(ctx->d_status);
  cudaFree(ctx->d_bar);
  cudaFree(ctx->d_keys);
  cudaFree(ctx->d_partials);
  cudaFree(ctx->d_H);
  cudaFree(ctx->d_Hb);
  cudaFree(ctx->d_Ab);
  cudaFree(ctx->d_gate_part);
  cudaFree(ctx->d_topk_part_i);
  cudaFree(ctx->d_v_lse_t);
  cudaFree(ctx->d_v_argmax_t);
  cudaFree(ctx->d_v_H);
  cudaFree(ctx->d_v_prev);
  cudaFree(ctx->d_v_rows);
  cudaFree(ctx->d_v_fail);
  cudaFree(ctx->d_v_count);
  cudaFree(ctx->d_l_prev);
  cudaFree(ctx->d_l_offq2);
  cudaFree(ctx->d_topk_part_v);
  delete ctx;
  return DSPARK_OK;
}

int dspark_ctx_reset(dspark_ctx* ctx, dspark_stream_t stream) {
  if (ctx == nullptr) return DSPARK_ERR_INVALID_ARG;
  if (cudaSetDevice(ctx->device) != cudaSuccess) return DSPARK_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  bool ok = cudaMemsetAsync(ctx->d_status, 0, sizeof(int), s) == cudaSuccess &&
            cudaMemsetAsync(ctx->d_bar, 0, sizeof(uint32_t), s) == cudaSuccess &&
            cudaMemsetAsync(ctx->d_keys, 0,
                            sizeof(unsigned long long) * ctx->K_max * dspark::kBatchChunk,
                            s) == cudaSuccess &&
            cudaMemsetAsync(ctx->d_v_fail, 0, sizeof(unsigned long long) * ctx->B_max, s) ==
                cudaSuccess &&
            cudaMemsetAsync(ctx->d_v_count, 0, sizeof(int) * ctx->B_max, s) == cudaSuccess;
  if (!ok) return DSPARK_ERR_CUDA;
  ctx->bar_counter = 0;
  ctx->epoch = 0;
  ctx->poisoned = 0;
  ctx->debug_skip_cta = -1;
  ctx->debug_refuse_launch = false;
  ctx->timeout_ns = dspark::kDefaultTimeoutNs;
  return DSPARK_OK;
}

int dspark_get_status(dspark_ctx* ctx, int* device_status) {
  if (ctx == nullptr || device_status == nullptr) return DSPARK_ERR_INVALID_ARG;
  if (cudaSetDevice(ctx->device) != cudaSuccess) return DSPARK_ERR_CUDA;
  int v = 0;
  if (cudaMemcpy(&v, ctx->d_status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
    return DSPARK_ERR_CUDA;
  *device_status = v;
  if (v != DSPARK_OK) ctx->poisoned = 1;
  return DSPARK_OK;
}

int dspark_debug_set(dspark_ctx* ctx, int cta, int timeout_ms) {
  if (ctx == nullptr) return DSPARK_ERR_INVALID_ARG;
  if (cta < -1) return DSPARK_ERR_INVALID_ARG;
  ctx->debug_skip_cta = cta;
  ctx->timeout_ns = timeout_ms > 0 ? static_cast<uint64_t>(timeout_ms) * 1000000ull
                                   : dspark::kDefaultTimeoutNs;
  return DSPARK_OK;
}

int dspark_debug_refuse_next_launch(dspark_ctx* ctx) {
  if (ctx == nullptr) return DSPARK_ERR_INVALID_ARG;
  ctx->debug_refuse_launch = true;
  return DSPARK_OK;
}

int dspark_last_launch_count(dspark_ctx* ctx) { return ctx ? ctx->last_launches : -1; }

int dspark_debug_trace(dspark_ctx* ctx, unsigned long long* device_buffer, int64_t capacity) {
  if (ctx == nullptr || (device_buffer == nullptr && capacity != 0) || capacity < 0)
    return DSPARK_ERR_INVALID_ARG;
  if (device_buffer != nullptr && (reinterpret_cast<uintptr_t>(device_buffer) & 7u) != 0)
    return DSPARK_ERR_INVALID_ARG;
  ctx->trace = device_buffer;
  ctx->trace_capacity = capacity;
  return DSPARK_OK;
}

int dspark_markov_draft(dspark_ctx* ctx, const float* U, const uint16_t* W1, const uint16_t* W2,
                        const int32_t* anchors, int B, int K, int V, int r, float temperature,
                        uint64_t seed, int32_t* tokens, float* logprobs,
                        const dspark_conf_args* conf, dspark_stream_t stream) {
  int st = check_draft_args(U, W1, W2, anchors, B, K, V, r, temperature, tokens, logprobs);
  if (st != DSPARK_OK) return st;
  st = check_conf(conf, r);
  if (st != DSPARK_OK) return st;
  if ((st = check_ctx(ctx)) != DSPARK_OK) return st;
  if (K > ctx->K_max || V > ctx->V_max) return DSPARK_ERR_CAPACITY;
  ctx->last_launches = 0;
  return run_draft(ctx, temperature > 0.f ? dspark::kModeSample : dspark::kModeGreedy, U, W1, W2,
                   anchors, nullptr, nullptr, B, K, V, r, temperature, seed, tokens, logprobs,
                   nullptr, nullptr, conf, reinterpret_cast<cudaStream_t>(stream));
}

int dspark_gated_draft(dspark_ctx* ctx, const float* U, const uint16_t* W1, const uint16_t* W2,
                       const int32_t* anchors, const uint16_t* h, const uint16_t* Wg, int d,
                       int B, int K, int V, int r, float temperature, uint64_t seed,
                       int32_t* tokens, float* logprobs, const dspark_conf_args* conf,
                       dspark_stream_t stream) {
  int st = check_draft_args(U, W1, W2, anchors, B, K, V, r, temperature, tokens, logprobs);
  if (st != DSPARK_OK) return st;
  if ((st = check_gate_args(h, Wg, d, r)) != DSPARK_OK) return st;
  if ((st = check_conf(conf, r)) != DSPARK_OK) return st;
  if ((st = check_ctx(ctx)) != DSPARK_OK) return st;
  if (K > ctx->K_max || V > ctx->V_max ||
      static_cast<int64_t>(B) * K > static_cast<int64_t>(ctx->B_max) * ctx->K_max)
    return DSPARK_ERR_CAPACITY;
  ctx->last_launches = 0;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  st = run_gate(ctx, h, Wg, B * K, d, r, nullptr, ctx->d_Hb, s);
  if (st != DSPARK_OK) return st;
  return run_draft(ctx, temperature > 0.f ? dspark::kModeSample : dspark::kModeGreedy, U, W1, W2,
                   anchors, nullptr, ctx->d_Hb, B, K, V, r, temperature, seed, tokens, logprobs,
                   nullptr, nullptr, conf, s);
}

int dspark_gate(dspark_ctx* ctx, const uint16_t* h, const uint16_t* Wg, int M, int d, int r,
                float* H, dspark_stream_t stream) {
  int st = check_gate_args(h, Wg, d, r);
  if (st != DSPARK_OK) return st;
  if (H == nullptr || M <= 0) return DSPARK_ERR_INVALID_ARG;
  if (!aligned16(H)) return DSPARK_ERR_INVALID_ARG;
  if ((st = check_ctx(ctx)) != DSPARK_OK) return st;
  if (static_cast<int64_t>(M) > static_cast<int64_t>(ctx->B_max) * ctx->K_max)
    return DSPARK_ERR_CAPACITY;
  ctx->last_launches = 0;
  return run_gate(ctx, h, Wg, M, d, r, H, nullptr, reinterpret_cast<cudaStream_t>(stream));
}

int dspark_selector_scores(dspark_ctx* ctx, const float* U, const uint16_t* A,
                           const uint16_t* Bt, const int32_t* anchors, const uint16_t* h,
                           const uint16_t* Wg, int d, int B, int K, int V, int r, int topk,
                           int32_t* cand, float* cand_U, float* scores, dspark_stream_t stream) {
  if (U == nullptr || A == nullptr || Bt == nullptr || anchors == nullptr || cand == nullptr ||
      cand_U == nullptr || scores == nullptr)
    return DSPARK_ERR_INVALID_ARG;
  if (B <= 0 || K <= 0 || V <= 0 || r <= 0 || topk <= 0) return DSPARK_ERR_INVALID_ARG;
  if (topk > dspark::kMaxTopk || topk > V || (V % 4) != 0 || K > dspark::kMaxK ||
      (r % 16) != 0 || r > dspark::kMaxRank)
    return DSPARK_ERR_UNSUPPORTED;
  const bool gated = (h != nullptr) || (Wg != nullptr);
  int st;
  if (gated && (st = check_gate_args(h, Wg, d, r)) != DSPARK_OK) return st;
  if (!aligned16(U) || !aligned16(A) || !aligned16(Bt)) return DSPARK_ERR_INVALID_ARG;
  if ((st = check_ctx(ctx)) != DSPARK_OK) return st;
  if (gated && static_cast<int64_t>(B) * K > static_cast<int64_t>(ctx->B_max) * ctx->K_max)
    return DSPARK_ERR_CAPACITY;
  ctx->last_launches = 0;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int n_topk = 0;
  cudaError_t e = dspark::launch_topk(U, B * K, V, topk, cand, cand_U, ctx->d_topk_part_i,
                                      ctx->d_topk_part_v, dspark::kTopkPartUnits, ctx->d_status,
                                      ctx->timeout_ns, &n_topk, s);
  ctx->last_launches += n_topk;
  if (e != cudaSuccess) return DSPARK_ERR_CUDA;
  if (gated) {
    st = run_gate(ctx, h, Wg, B * K, d, r, ctx->d_H, nullptr, s);
    if (st != DSPARK_OK) return st;
  }
  e = dspark::launch_pair_scores(cand, cand_U, A, Bt, anchors, gated ? ctx->d_H : nullptr, B, K,
                                 V, r, topk, scores, ctx->d_status, ctx->timeout_ns, s);
  ctx->last_launches += 1;
  return cuda_status(e);
}

int dspark_selector_walk(dspark_ctx* ctx, const int32_t* cand, const float* scores,
                         const int32_t* anchors, const uint16_t* A, int B, int K, int V, int r,
                         int topk, float temperature, uint64_t seed, int32_t* tokens,
                         float* logprobs, const dspark_conf_args* conf, dspark_stream_t stream) {
  if (cand == nullptr || scores == nullptr || tokens == nullptr || logprobs == nullptr ||
      anchors == nullptr)
    return DSPARK_ERR_INVALID_ARG;
  if (B <= 0 || K <= 0 || V <= 0 || topk <= 0) return DSPARK_ERR_INVALID_ARG;
  if (topk > dspark::kMaxTopk || topk > V || K > dspark::kMaxK) return DSPARK_ERR_UNSUPPORTED;
  if (!(temperature >= 0.f) || temperature > 3.0e38f) return DSPARK_ERR_INVALID_ARG;
  int st;
  if (conf != nullptr) {
    if ((st = check_conf(conf, r)) != DSPARK_OK) return st;
    if (conf->with_markov &&
        (A == nullptr || !aligned16(A) || r <= 0 || (r % 8) != 0 || r > dspark::kMaxRank))
      return DSPARK_ERR_INVALID_ARG;
  }
  if ((st = check_ctx(ctx)) != DSPARK_OK) return st;
  ctx->last_launches = 0;
  const float inv_t = temperature > 0.f ? 1.0f / temperature : 1.0f;
  cudaError_t e = dspark::launch_walk(cand, scores, anchors, A, B, K, V, r, topk, inv_t,
                                      temperature > 0.f ? 1 : 0,
                                      static_cast<uint32_t>(seed & 0xFFFFFFFFull),
                                      static_cast<uint32_t>(seed >> 32), tokens, logprobs, conf,
                                      ctx->d_status, reinterpret_cast<cudaStream_t>(stream));
  ctx->last_launches += 1;
  return cuda_status(e);
}

int dspark_confidence(dspark_ctx* ctx, const uint16_t* h, const uint16_t* W1,
                      const int32_t* anchors, const int32_t* tokens, const uint16_t* w,
                      float bias, int with_markov, int B, int K, int d, int r, int V,
                      float threshold, const float* tau, float* conf, float* cumprod,
                      int32_t* verify_len, dspark_stream_t stream) {
  if (h == nullptr || w == nullptr || conf == nullptr || cumprod == nullptr ||
      verify_len == nullptr)
    return DSPARK_ERR_INVALID_ARG;
  if (B <= 0 || K <= 0 || d <= 0 || (d % 8) != 0) return DSPARK_ERR_INVALID_ARG;
  if (K > dspark::kMaxK) return DSPARK_ERR_UNSUPPORTED;
  if (with_markov) {
    if (W1 == nullptr || anchors == nullptr || tokens == nullptr || V <= 0)
      return DSPARK_ERR_INVALID_ARG;
    if (r <= 0 || (r % 8) != 0 || r > dspark::kMaxRank) return DSPARK_ERR_INVALID_ARG;
    if (!aligned16(W1)) return DSPARK_ERR_INVALID_ARG;
  }
  if (!aligned16(h) || !aligned16(w) || !(threshold == threshold)) return DSPARK_ERR_INVALID_ARG;
  int st;
  if ((st = check_ctx(ctx)) != DSPARK_OK) return st;
  ctx->last_launches = 1;
  return cuda_status(dspark::launch_confidence(h, W1, anchors, tokens, w, bias, with_markov, B, K,
                                               d, with_markov ? r : 0, V, threshold, tau, conf,
                                               cumprod, verify_len, ctx->d_status,
                                               reinterpret_cast<cudaStream_t>(stream)));
}

int dspark_markov_logits(dspark_ctx* ctx, const float* U, const uint16_t* W1, const uint16_t* W2,
                         const int32_t* prev_tokens, const uint16_t* h, const uint16_t* Wg,
                         int d, int B, int K, int V, int r, float temperature, float* logits,
                         float* lse, dspark_stream_t stream) {
  if (prev_tokens == nullptr) return DSPARK_ERR_INVALID_ARG;
  int st = check_draft_args(U, W1, W2, prev_tokens, B, K, V, r, temperature, logits, lse);
  if (st != DSPARK_OK) return st;
  const bool gated = (h != nullptr) || (Wg != nullptr);
  if (gated && (st = check_gate_args(h, Wg, d, r)) != DSPARK_OK) return st;
  if (!aligned16(logits)) return DSPARK_ERR_INVALID_ARG;
  if ((st = check_ctx(ctx)) != DSPARK_OK) return st;
  if (K > ctx->K_max || V > ctx->V_max) return DSPARK_ERR_CAPACITY;
  if (gated && static_cast<int64_t>(B) * K > static_cast<int64_t>(ctx->B_max) * ctx->K_max)
    return DSPARK_ERR_CAPACITY;
  ctx->last_launches = 0;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (gated) {
    st = run_gate(ctx, h, Wg, B * K, d, r, nullptr, ctx->d_Hb, s);
    if (st != DSPARK_OK) return st;
  }
  return run_draft(ctx, dspark::kModeTeacherForced, U, W1, W2, prev_tokens, prev_tokens,
                   gated ? ctx->d_Hb : nullptr, B, K, V, r, temperature, 0, nullptr, nullptr,
                   logits, lse, nullptr, s);
}

int dspark_rnn_draft(dspark_ctx* ctx, const float* U, const uint16_t* W1, const uint16_t* W2,
                     const int32_t* anchors, const uint16_t* h, const uint16_t* Wa,
                     const uint16_t* Wg, int d, int B, int K, int V, int r, float temperature,
                     uint64_t seed, int32_t* tokens, float* logprobs,
                     const dspark_conf_args* conf, dspark_stream_t stream) {
  int st = check_draft_args(U, W1, W2, anchors, B, K, V, r, temperature, tokens, logprobs);
  if (st != DSPARK_OK) return st;
  if ((st = check_rnn_args(h, Wa, Wg, d, r)) != DSPARK_OK) return st;
  if ((st = check_conf(conf, r)) != DSPARK_OK) return st;
  if ((st = check_ctx(ctx)) != DSPARK_OK) return st;
  if (K > ctx->K_max || V > ctx->V_max ||
      static_cast<int64_t>(B) * K > static_cast<int64_t>(ctx->B_max) * ctx->K_max)
    return DSPARK_ERR_CAPACITY;
  ctx->last_launches = 0;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const uint16_t* H = nullptr;
  if ((st = run_rnn_gates(ctx, h, Wa, Wg, B * K, d, r, &H, s)) != DSPARK_OK) return st;
  return run_draft(ctx, temperature > 0.f ? dspark::kModeSample : dspark::kModeGreedy, U, W1, W2,
                   anchors, nullptr, H, B, K, V, r, temperature, seed, tokens, logprobs, nullptr,
                   nullptr, conf, s, nullptr, ctx->d_Ab);
}

int dspark_rnn_logits(dspark_ctx* ctx, const float* U, const uint16_t* W1, const uint16_t* W2,
                      const int32_t* prev_tokens, const uint16_t* h, const uint16_t* Wa,
                      const uint16_t* Wg, int d, int B, int K, int V, int r, float temperature,
                      float* logits, float* lse, dspark_stream_t stream) {
  if (prev_tokens == nullptr) return DSPARK_ERR_INVALID_ARG;
  int st = check_draft_args(U, W1, W2, prev_tokens, B, K, V, r, temperature, logits, lse);
  if (st != DSPARK_OK) return st;
  if ((st = check_rnn_args(h, Wa, Wg, d, r)) != DSPARK_OK) return st;
  if (!aligned16(logits)) return DSPARK_ERR_INVALID_ARG;
  if ((st = check_ctx(ctx)) != DSPARK_OK) return st;
  if (K > ctx->K_max || V > ctx->V_max ||
      static_cast<int64_t>(B) * K > static_cast<int64_t>(ctx->B_max) * ctx->K_max)
    return DSPARK_ERR_CAPACITY;
  ctx->last_launches = 0;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const uint16_t* H = nullptr;
  if ((st = run_rnn_gates(ctx, h, Wa, Wg, B * K, d, r, &H, s)) != DSPARK_OK) return st;
  return run_draft(ctx, dspark::kModeTeacherForced, U, W1, W2, prev_tokens, prev_tokens, H, B, K,
                   V, r, temperature, 0, nullptr, nullptr, logits, lse, nullptr, s, nullptr,
                   ctx->d_Ab);
}

int dspark_verify(dspark_ctx* ctx, const float* P, const float* U, const uint16_t* W1,
                  const uint16_t* W2, const int32_t* anchors, const uint16_t* h,
                  const uint16_t* Wg, int d, const int32_t* tokens, const float* draft_logprobs,
                  const int32_t* ell, int B, int K, int V, int r, float draft_temperature,
                  float target_temperature, uint64_t seed, int32_t* n_acc, int32_t* next_token,
                  float* accept_prob, dspark_stream_t stream) {
  if (P == nullptr || tokens == nullptr || n_acc == nullptr || next_token == nullptr)
    return DSPARK_ERR_INVALID_ARG;
  int st = check_draft_args(U, W1, W2, anchors, B, K, V, r, draft_temperature, n_acc, next_token);
  if (st != DSPARK_OK) return st;
  if (!(target_temperature >= 0.f) || target_temperature > 3.0e38f) return DSPARK_ERR_INVALID_ARG;
  if (draft_temperature > 0.f && draft_logprobs == nullptr) return DSPARK_ERR_INVALID_ARG;
  if (!aligned16(P)) return DSPARK_ERR_INVALID_ARG;
  const bool gated = (h != nullptr) || (Wg != nullptr);
  if (gated && (st = check_gate_args(h, Wg, d, r)) != DSPARK_OK) return st;
  if ((st = check_ctx(ctx)) != DSPARK_OK) return st;
  if (B > ctx->B_max || K > ctx->K_max || V > ctx->V_max) return DSPARK_ERR_CAPACITY;
  ctx->last_launches = 0;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (gated) {
    st = run_gate(ctx, h, Wg, B * K, d, r, ctx->d_H, nullptr, s);
    if (st != DSPARK_OK) return st;
  }
  dspark::VerifyArgs v{};
  v.P = P;
  v.U = U;
  v.W1 = W1;
  v.W2 = W2;
  v.H = gated ? ctx->d_H : nullptr;
  v.tokens = tokens;
  v.logq = draft_logprobs;
  v.anchors = anchors;
  v.ell = ell;
  v.B = B;
  v.K = K;
  v.V = V;
  v.r = r;
  v.draft_temperature = draft_temperature;
  v.target_temperature = target_temperature;
  v.seed_lo = static_cast<uint32_t>(seed & 0xFFFFFFFFull);
  v.seed_hi = static_cast<uint32_t>(seed >> 32);
  v.n_acc = n_acc;
  v.next_token = next_token;
  v.accept_prob = accept_prob;
  v.status = ctx->d_status;
  v.lse_t = ctx->d_v_lse_t;
  v.argmax_t = ctx->d_v_argmax_t;
  v.H_sel = ctx->d_v_H;
  v.prev_sel = ctx->d_v_prev;
  v.rows = target_temperature > 0.f ? ctx->d_v_rows : nullptr;
  v.fail_mask = ctx->d_v_fail;
  v.count = ctx->d_v_count;
  int n = 0;
  cudaError_t e = dspark::launch_verify(v, s, &n);
  ctx->last_launches += n;
  if (e != cudaSuccess) return DSPARK_ERR_CUDA;
  if (target_temperature > 0.f) {
    // the draw: the draft kernel's residual mode over one position, reading each request's
    // draw rows of U and P in place (a greedy target's token is its argmax, set above)
    LabelIn res{P, nullptr, nullptr, nullptr, 1.4426950408889634f / target_temperature,
                ctx->d_v_rows, K};
    st = run_draft(ctx, dspark::kModeResidual, U, W1, W2, ctx->d_v_prev, ctx->d_v_prev,
                   gated ? ctx->d_v_H : nullptr, B, 1, V, r, draft_temperature, seed, next_token,
                   nullptr, nullptr, nullptr, nullptr, s, &res);
    if (st != DSPARK_OK) return st;
  }
  return DSPARK_OK;
}

int dspark_accept_label(dspark_ctx* ctx, const float* P, const float* U, const uint16_t* W1,
                        const uint16_t* W2, const int32_t* anchors, const uint16_t* h,
                        const uint16_t* Wg, int d, const int32_t* tokens,
                        const float* draft_logprobs, int B, int K, int V, int r,
                        float draft_temperature, float target_temperature, float* label,
                        dspark_stream_t stream) {
  if (P == nullptr) return DSPARK_ERR_INVALID_ARG;
  int st = check_draft_args(U, W1, W2, anchors, B, K, V, r, draft_temperature, tokens, label);
  if (st != DSPARK_OK) return st;
  if (!(target_temperature >= 0.f) || target_temperature > 3.0e38f) return DSPARK_ERR_INVALID_ARG;
  if (draft_temperature > 0.f && draft_logprobs == nullptr) return DSPARK_ERR_INVALID_ARG;
  if (!aligned16(P)) return DSPARK_ERR_INVALID_ARG;
  const bool gated = (h != nullptr) || (Wg != nullptr);
  if (gated && (st = check_gate_args(h, Wg, d, r)) != DSPARK_OK) return st;
  if ((st = check_ctx(ctx)) != DSPARK_OK) return st;
  if (B > ctx->B_max || K > ctx->K_max || V > ctx->V_max) return DSPARK_ERR_CAPACITY;
  ctx->last_launches = 0;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (gated) {
    st = run_gate(ctx, h, Wg, B * K, d, r, ctx->d_H, ctx->d_Hb, s);
    if (st != DSPARK_OK) return st;
  }
  // the target's normaliser (or argmax) of rows k < K and each row's preparation
  dspark::LabelPrepArgs a{};
  a.P = P;
  a.U = U;
  a.W1 = W1;
  a.W2 = W2;
  a.H = gated ? ctx->d_H : nullptr;
  a.anchors = anchors;
  a.tokens = tokens;
  a.logq = draft_logprobs;
  a.lse_t = ctx->d_v_lse_t;
  a.argmax_t = ctx->d_v_argmax_t;
  a.B = B;
  a.K = K;
  a.V = V;
  a.r = r;
  a.inv_td = draft_temperature > 0.f ? 1.0f / draft_temperature : 0.f;
  a.inv_tt = target_temperature > 0.f ? 1.0f / target_temperature : 0.f;
  a.prev = ctx->d_l_prev;
  a.offq2 = ctx->d_l_offq2;
  a.label = label;
  a.status = ctx->d_status;
  if (dspark::launch_label_prep(a, s) != cudaSuccess) return DSPARK_ERR_CUDA;
  ctx->last_launches += 1;
  if (draft_temperature > 0.f && target_temperature > 0.f) {
    LabelIn lab{P, ctx->d_v_lse_t, ctx->d_l_offq2, label,
                1.4426950408889634f / target_temperature, nullptr};
    st = run_draft(ctx, dspark::kModeLabel, U, W1, W2, anchors, ctx->d_l_prev,
                   gated ? ctx->d_Hb : nullptr, B, K, V, r, draft_temperature, 0, nullptr, nullptr,
                   nullptr, nullptr, nullptr, s, &lab);
    if (st != DSPARK_OK) return st;
  }
  return DSPARK_OK;
}

int dspark_sts_fit(dspark_ctx* ctx, const float* conf, const float* label, int N, int K,
                   float tau_lo, float tau_hi, float* tau, float* loss, dspark_stream_t stream) {
  if (conf == nullptr || label == nullptr || tau == nullptr) return DSPARK_ERR_INVALID_ARG;
  if (N <= 0 || K <= 0 || !(tau_lo > 0.f) || !(tau_hi > tau_lo) || tau_hi > 3.0e38f)
    return DSPARK_ERR_INVALID_ARG;
  if (K > dspark::kMaxK) return DSPARK_ERR_UNSUPPORTED;
  int st;
  if ((st = check_ctx(ctx)) != DSPARK_OK) return st;
  ctx->last_launches = 1;
  return cuda_status(dspark::launch_sts_fit(conf, label, N, K, tau_lo, tau_hi, tau, loss,
                                            reinterpret_cast<cudaStream_t>(stream)));
}

int dspark_schedule(dspark_ctx* ctx, const float* a, int R, int K, const float* sps,
                    int sps_len, int32_t* ell, float* theta, dspark_stream_t stream) {
  if ((a == nullptr && K > 0) || sps == nullptr || ell == nullptr) return DSPARK_ERR_INVALID_ARG;
  if (R <= 0 || K < 0) return DSPARK_ERR_INVALID_ARG;
  if (static_cast<int64_t>(R) * K > dspark::kScheduleMaxCandidates || R > 65535 || K > 65535)
    return DSPARK_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(sps_len) < static_cast<int64_t>(R) * (K + 1) + 1)
    return DSPARK_ERR_INVALID_ARG;
  int st;
  if ((st = check_ctx(ctx)) != DSPARK_OK) return st;
  ctx->last_launches = 0;
  cudaError_t e = dspark::launch_schedule(a, R, K, sps, ell, theta,
                                          reinterpret_cast<cudaStream_t>(stream));
  ctx->last_launches = 1;
  return cuda_status(e);
}

}  // extern "C"
