// attn_diag.cu -- diagnostic kernels used by the tests.
//
// attn_diag_tile_kernel runs the fused kernel's two tensor-core products on a
// single tile, with the same shared-memory descriptors, instruction
// descriptors and tensor-memory layout:
//   S = Q K^T  (SS form: Q and K staged by TMA with 128-byte swizzle)
//   O = P V    (TS form: P written to tensor memory by the threads, V staged
//               by TMA, MN-major)
// and copies both accumulators back to global memory, so the building blocks
// can be checked against a host reference in isolation.
//
// attn_diag_wait_kernel waits on an mbarrier that never completes, bounded by
// a short limit, and records a timeout: the failure path of every bounded
// wait, exercised without faulting the GPU.
#include <cuda_bf16.h>

#include "attn_internal.cuh"
#include "ptx.cuh"

namespace attn {
namespace {

using namespace ptx;

constexpr uint32_t TILE = 128 * 64 * 2;  // 16 KB

struct __align__(1024) DiagSmem {
  uint8_t q[TILE];
  uint8_t k[TILE];
  uint8_t v[TILE];
  uint64_t tma_bar;
  uint64_t mma_bar;
  uint32_t tmem_base;
  int abort;
};

__global__ void __launch_bounds__(128, 1)
    attn_diag_tile_kernel(const __grid_constant__ CUtensorMap tmq,
                          const __grid_constant__ CUtensorMap tmk,
                          const __grid_constant__ CUtensorMap tmv, const uint32_t* p_packed,
                          float* s_out, float* o_out, uint64_t limit_ns, int* status) {
  extern __shared__ uint8_t smem_raw[];
  DiagSmem& sm = *reinterpret_cast<DiagSmem*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5;
  const int t = threadIdx.x;
  // S [0,128), O [128,192), P [192,256)
  constexpr uint32_t COL_S = 0, COL_O = 128, COL_P = 192;

  if (t == 0) {
    mbar_init(smem_u32(&sm.tma_bar), 1);
    mbar_init(smem_u32(&sm.mma_bar), 1);
    sm.abort = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(&sm.tmem_base), 256);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;

  if (t == 0) {
    const uint32_t bar = smem_u32(&sm.tma_bar);
    mbar_arrive_expect_tx(bar, 3 * TILE);
    tma_load_2d(smem_u32(sm.q), &tmq, bar, 0, 0);
    tma_load_2d(smem_u32(sm.k), &tmk, bar, 0, 0);
    tma_load_2d(smem_u32(sm.v), &tmv, bar, 0, 0);
  }
  // row t of P (128 bf16 = 64 packed words) into tensor-memory lane t
  {
    uint32_t a[32], b[32];
    const uint32_t* src = p_packed + static_cast<size_t>(t) * 64;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      a[i] = src[i];
      b[i] = src[32 + i];
    }
    tmem_st32(tmem + lane_off + COL_P, a);
    tmem_st32(tmem + lane_off + COL_P + 32, b);
    tmem_st_wait();
  }
  tc_fence_before();
  __syncthreads();

  bool ok = true;
  if (t == 0) {
    const int never = 0;
    ok = mbar_wait(smem_u32(&sm.tma_bar), 0, limit_ns, &never);
    tc_fence_after();
    if (ok) {
      constexpr uint32_t IDESC_S = idesc_bf16_f32(128, 128, false, false);
      constexpr uint32_t IDESC_O = idesc_bf16_f32(128, 64, false, true);
      const uint32_t qb = smem_u32(sm.q), kb = smem_u32(sm.k), vb = smem_u32(sm.v);
      for (int kk = 0; kk < 4; ++kk)
        mma_ss(tmem + COL_S, sdesc_sw128(qb + kk * 32, 16, 1024),
               sdesc_sw128(kb + kk * 32, 16, 1024), IDESC_S, kk > 0);
      for (int kk = 0; kk < 8; ++kk)
        mma_ts(tmem + COL_O, tmem + COL_P + kk * 8, sdesc_sw128(vb + kk * 16 * 128, 1024, 1024),
               IDESC_O, kk > 0);
    }
    tc_commit(smem_u32(&sm.mma_bar));
    if (!ok) {
      atomicCAS(status, kDevOk, kDevTimeout);
      sm.abort = 1;
    }
  }
  __syncthreads();
  {
    const int never = 0;
    ok = mbar_wait(smem_u32(&sm.mma_bar), 0, limit_ns, &never);
    ok = __all_sync(0xffffffffu, ok) && !sm.abort;
    tc_fence_after();
    if (ok) {
      uint32_t r[32];
      for (int c = 0; c < 128; c += 32) {
        tmem_ld32(tmem + lane_off + COL_S + c, r);
        tmem_ld_wait(r);
        for (int i = 0; i < 32; ++i) s_out[t * 128 + c + i] = __uint_as_float(r[i]);
      }
      for (int c = 0; c < 64; c += 32) {
        tmem_ld32(tmem + lane_off + COL_O + c, r);
        tmem_ld_wait(r);
        for (int i = 0; i < 32; ++i) o_out[t * 64 + c + i] = __uint_as_float(r[i]);
      }
    } else if (t == 0) {
      atomicCAS(status, kDevOk, kDevTimeout);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 256);
  }
}

__global__ void attn_diag_wait_kernel(uint64_t limit_ns, int* status) {
  __shared__ uint64_t bar;
  const int never = 0;
  mbar_init(smem_u32(&bar), 1);
  fence_mbar_init();
  // Nobody arrives on `bar`: phase 0 never completes.
  if (!mbar_wait(smem_u32(&bar), 0, limit_ns, &never)) atomicCAS(status, kDevOk, kDevTimeout);
}

}  // namespace

cudaError_t launch_diag_tile(const CUtensorMap& tmq, const CUtensorMap& tmk,
                             const CUtensorMap& tmv, const void* p, float* s, float* o,
                             const LaunchCtx& ctx) {
  const size_t smem = sizeof(DiagSmem) + 1024;
  cudaError_t err = cudaFuncSetAttribute(
      attn_diag_tile_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (err != cudaSuccess) return err;
  attn_diag_tile_kernel<<<1, 128, smem, ctx.stream>>>(
      tmq, tmk, tmv, static_cast<const uint32_t*>(p), s, o, ctx.limit_ns, ctx.status);
  return cudaGetLastError();
}

cudaError_t launch_diag_wait_timeout(uint64_t limit_ns, const LaunchCtx& ctx) {
  attn_diag_wait_kernel<<<1, 1, 0, ctx.stream>>>(limit_ns, ctx.status);
  return cudaGetLastError();
}

}  // namespace attn
