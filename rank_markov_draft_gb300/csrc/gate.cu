// gate.cu -- gate prologue of the gated Markov head: H = sigmoid(h . Wg).
//
// Source: equivalence page, "What the two methods do" (the context-dependent
// gate H(h_t) is computed from the current hidden state) and "The
// equivalence..." (gated rule logits_t = U_t + (W1[a] (.) H(h_t))^T W2).
// The pages leave H's form open; this library reads it as a linear map of
// h_t followed by a logistic sigmoid, without bias.
//
// No position depends on a sampled token, so the whole block's gate is one
// dense GEMM [B*K, d] x [d, r] run before the draft: tcgen05.mma with TMA-fed
// 128B-swizzled tiles (h K-major, Wg MN-major, fp32 accumulator in TMEM).
// The reduction over d is split across CTAs to fill the GPU; each split
// writes its own fp32 partial and a finaliser sums them in a fixed order and
// applies the sigmoid, so results do not depend on scheduling.

#include <algorithm>
#include <cstdint>
#include <cuda_bf16.h>

#include "internal.h"
#include "sm103.cuh"

namespace dspark {
namespace {

constexpr int kStages = 8;  // 192 KB of h and Wg in flight: the fills are L2-latency bound
constexpr uint32_t kAStage = 128 * 64 * 2;  // 16 KB: 128 rows of h x 64 of d
constexpr uint32_t kBStage = 64 * 64 * 2;   // 8 KB: 64 of d x 64 of r
constexpr uint32_t kOffA = 0;
constexpr uint32_t kOffB = kOffA + kStages * kAStage;
constexpr uint32_t kOffBar = kOffB + kStages * kBStage;
constexpr uint32_t kSmem = kOffBar + 256 + 1024;
constexpr int kThreads = 192;  // producer, MMA, 4 epilogue warps
constexpr uint32_t kTmemCols = 64;

__global__ void __launch_bounds__(kThreads, 1) gate_gemm_kernel(const __grid_constant__ GateArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem + kOffA;
  uint8_t* sB = smem + kOffB;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint64_t* full = bars;               // [kStages]
  uint64_t* empty = bars + kStages;    // [kStages]
  uint64_t* acc_full = bars + 2 * kStages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * kStages + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 2 * kStages + 2);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m0 = blockIdx.x * 128, n0 = blockIdx.y * 64, split = blockIdx.z;
  const int nchunks = a.d / 64;
  const int c_begin = split * a.chunks_per_split;
  const int c_end = min(nchunks, c_begin + a.chunks_per_split);
  const int nc = c_end - c_begin;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(acc_full, 1);
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&a.tm_h);
    tma_prefetch_desc(&a.tm_wg);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      const uint64_t pol = l2_policy_evict_first();
      const uint64_t pol_w = l2_policy_evict_last();
      bool ok = true;
      int issued = 0;
      for (int i = 0; i < nc; ++i) {
        const int s = i % kStages;
        if (!mbar_wait(&empty[s], ((i / kStages) & 1) ^ 1, a.timeout_ns, abort_flag)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(&full[s], kAStage + kBStage);
        tma_load_2d(sA + s * kAStage, &a.tm_h, (c_begin + i) * 64, m0, &full[s], pol);
        tma_load_2d(sB + s * kBStage, &a.tm_wg, n0, (c_begin + i) * 64, &full[s], pol_w);
        issued = i + 1;
      }
      if (!ok) {
        *abort_flag = 1;
        record_error(a.status, kStatusTimeout);
        for (int i = issued - 1; i >= 0 && i >= issued - kStages; --i)
          mbar_wait(&full[i % kStages], (i / kStages) & 1, a.timeout_ns, nullptr);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(128, 64, /*a_mn=*/false, /*b_mn=*/true);
      bool ok = true;
      bool issued_any = false;
      for (int i = 0; i < nc; ++i) {
        const int s = i % kStages;
        if (!mbar_wait(&full[s], (i / kStages) & 1, a.timeout_ns, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t a0 = smem_addr(sA + s * kAStage), b0 = smem_addr(sB + s * kBStage);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          umma_bf16(tmem, smem_desc(a0 + kk * 32, 16, 1024), smem_desc(b0 + kk * 2048, 1024, 1024),
                    idesc, (i > 0 || kk > 0) ? 1u : 0u);
        }
        umma_commit(&empty[s]);
        issued_any = true;
      }
      if (!ok) {
        *abort_flag = 1;
        record_error(a.status, kStatusTimeout);
      }
      if (issued_any) {
        umma_commit(acc_full);
      } else {
        mbar_arrive(acc_full);
      }
    }
  } else {
    const int q = warp & 3;
    const bool ok = __all_sync(0xFFFFFFFFu, mbar_wait(acc_full, 0, a.timeout_ns, nullptr));
    if (!ok) {
      record_error(a.status, kStatusTimeout);
    } else if (!*abort_flag) {
      tc_fence_after();
      const int row = m0 + q * 32 + lane;
      float* dst = a.partial + (static_cast<size_t>(split) * a.M + row) * a.r + n0;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t v[16];
        tmem_ld_x16(tmem + (static_cast<uint32_t>(q * 32) << 16) + c * 16, v);
        tmem_wait_ld();
        if (row < a.M) {
          float4* d4 = reinterpret_cast<float4*>(dst + c * 16);
#pragma unroll
          for (int j = 0; j < 4; ++j)
            d4[j] = make_float4(__uint_as_float(v[4 * j]), __uint_as_float(v[4 * j + 1]),
                                __uint_as_float(v[4 * j + 2]), __uint_as_float(v[4 * j + 3]));
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// H = sigmoid(sum over splits, in split order); n4 float4 per split, all of a
// thread's split loads in flight before the sum.  H (fp32) and Hb (the same values
// rounded to bf16, for the draft kernel's packed operand arithmetic) are each optional.
__global__ void gate_finalize_kernel(const float4* __restrict__ partial, int splits, int64_t n4,
                                     float4* __restrict__ H, uint2* __restrict__ Hb) {
  // a draft launched as this kernel's programmatic dependent may start its prologue now
  griddep_launch_dependents();
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n4;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    float4 pv[8];
#pragma unroll
    for (int s = 0; s < 8; ++s)
      pv[s] = (s < splits) ? __ldcs(partial + s * n4 + i) : make_float4(0.f, 0.f, 0.f, 0.f);
    float4 z = pv[0];
#pragma unroll
    for (int s = 1; s < 8; ++s) {
      z.x += pv[s].x;
      z.y += pv[s].y;
      z.z += pv[s].z;
      z.w += pv[s].w;
    }
    const float4 g = make_float4(1.0f / (1.0f + expf(-z.x)), 1.0f / (1.0f + expf(-z.y)),
                                 1.0f / (1.0f + expf(-z.z)), 1.0f / (1.0f + expf(-z.w)));
    if (H != nullptr) H[i] = g;
    if (Hb != nullptr) {
      const __nv_bfloat162 lo = __floats2bfloat162_rn(g.x, g.y);
      const __nv_bfloat162 hi = __floats2bfloat162_rn(g.z, g.w);
      Hb[i] = make_uint2(*reinterpret_cast<const uint32_t*>(&lo),
                         *reinterpret_cast<const uint32_t*>(&hi));
    }
  }
}

}  // namespace

cudaError_t launch_gate_gemm(const GateArgs& args, cudaStream_t stream) {
  cudaError_t err = cudaFuncSetAttribute(reinterpret_cast<const void*>(&gate_gemm_kernel),
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kSmem));
  if (err != cudaSuccess) return err;
  dim3 grid((args.M + 127) / 128, args.r / 64, args.splits);
  gate_gemm_kernel<<<grid, kThreads, kSmem, stream>>>(args);
  return cudaGetLastError();
}

cudaError_t launch_gate_finalize(const float* partial, int splits, int64_t n, float* H,
                                 uint16_t* Hb, cudaStream_t stream) {
  // n = M * r is a multiple of 64 (r % 64 == 0) and splits <= 8
  const int64_t n4 = n / 4;
  int blocks = static_cast<int>(std::min<int64_t>((n4 + 255) / 256, 4096));
  if (blocks < 1) blocks = 1;
  gate_finalize_kernel<<<blocks, 256, 0, stream>>>(reinterpret_cast<const float4*>(partial), splits,
                                                   n4, reinterpret_cast<float4*>(H),
                                                   reinterpret_cast<uint2*>(Hb));
  return cudaGetLastError();
}

}  // namespace dspark
