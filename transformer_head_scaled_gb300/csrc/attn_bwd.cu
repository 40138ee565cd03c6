// attn_bwd.cu -- backward of the fused attention forward for sm_103a: the
// gradients dQ, dK, dV of a loss whose gradient with respect to the output
// O = softmax(scale * Q K^T + M) V is dO.
//
// The forward is eq. (1) of "Attention Is All You Need" (section 3.2.1) with
// the masks of section 3.2.3; its gradient is what training the model of
// section 5 back-propagates through every attention layer.  Per (b, h), with
// P the row softmax recomputed from Q, K and the forward's log-sum-exp:
//
//   dV = P^T dO,   dP = dO V^T,   D_i = sum_c dO_ic O_ic,
//   dS = P * (dP - D_i)  (elementwise),   dQ = scale dS K,   dK = scale dS^T Q.
//
// Three launches:
//   1. attn_bwd_pre_kernel: per query row, -D_i and -LSE_i * log2(e) into the
//      workspace (zero on the padding rows of each 128-row tile), and the row
//      of the fp32 dQ accumulator set to zero.
//   2. attn_bwd_tc_kernel: one persistent CTA per SM walks work items = one
//      128-key tile of one (b, h); for each 128-query tile that the mask lets
//      see those keys it runs the five tensor-core products of that tile pair
//      and accumulates dK and dV in tensor memory; dQ of the tile pair is
//      added into the fp32 accumulator in global memory with a TMA reduce.
//   3. attn_bwd_dq_kernel: dQ = scale * accumulator, rounded to bf16.
//
// Kernel 2 (448 threads):
//   warps 0-7   the elementwise part: warp w owns tensor-memory lanes
//               32*(w%4).. (= keys) and query columns 64*(w/4)..+63; it turns
//               S^T into P^T and dP^T into dS^T and writes both, as bf16, into
//               shared memory in the 128-byte swizzled layout the MMAs read;
//   warps 8-11  epilogue: dQ of each tile pair (tensor memory -> swizzled fp32
//               staging -> TMA reduce-add), dK and dV of each item (-> bf16 ->
//               TMA store);
//   warp  12    TMA producer: K, V per item (2 slots), Q, dO, -LSE2, -D per
//               query tile (2 stages);
//   warp  13    tensor-memory owner and MMA issuer.
// Tensor memory (512 columns): S^T [0,128)  dP^T [128,256)  dV [256,320)
// dK [320,384)  dQ [384,448).  Keys are the 128 lanes of S^T, dP^T, dV, dK;
// queries are the lanes of dQ.
// Per tile pair t the MMAs are issued in the order
//   dV(t), S^T(t+1), dP^T(t+1), dK(t), dQ(t)
// so that the elementwise warps can start on tile t+1 while the tensor pipe
// finishes the gradient products of tile t.  Every wait is bounded; on timeout
// the kernel records kDevTimeout, all roles drain and the CTA returns.
#include <cuda_bf16.h>

#include "attn_internal.cuh"
#include "ptx.cuh"

namespace attn {
namespace {

using namespace ptx;

constexpr int BM = 128;  // queries per query tile
constexpr int BN = 128;  // keys per key tile (= tensor-memory lanes)
constexpr int D = 64;    // head size
constexpr uint32_t TILE_BYTES = 128 * D * 2;  // a [128 x 64] bf16 tile: 16 KB
constexpr int NUM_THREADS = 448;
constexpr int EPI_WARP0 = 8;
constexpr int LOAD_WARP = 12;
constexpr int MMA_WARP = 13;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t COL_S = 0, COL_DP = 128, COL_DV = 256, COL_DK = 320, COL_DQ = 384;
constexpr int EPI_BAR = 1;  // named barrier of the 128 epilogue threads
constexpr float LOG2E = 1.4426950408889634f;

static_assert(BM == BN, "the causal tile range assumes square tiles");

struct __align__(1024) Smem {
  uint8_t k[2][TILE_BYTES];
  uint8_t v[2][TILE_BYTES];
  uint8_t q[2][TILE_BYTES];
  uint8_t dout[2][TILE_BYTES];
  // P^T and dS^T as [128 keys x 128 queries] bf16: two 64-query column blocks
  // of [128 x 64], each in the 128-byte swizzled layout.
  uint8_t pt[2][TILE_BYTES];
  uint8_t dst[2][TILE_BYTES];
  uint8_t stage[TILE_BYTES];  // epilogue staging (fp32 half of dQ, or bf16 dK / dV)
  float nlse2[2][BM];         // -LSE * log2(e) of the stage's queries
  float nd[2][BM];            // -D of the stage's queries
  uint64_t kv_full[2], kv_empty[2];
  uint64_t q_full[2], q_empty[2];
  uint64_t s_full, s_free, dp_full, dp_free;
  uint64_t p_full, p_free, ds_full, ds_free;
  uint64_t dq_full, dq_free, dkv_full, dkv_free;
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};

struct Params {
  const float* nlse2;  // [BH][nq_pad]
  const float* nd;     // [BH][nq_pad]
  const int* key_lens;
  int H, n_q, n_k, BH, nq_pad;
  int mask;
  int num_qt, num_kt, num_items;
  float scale_log2;  // scale * log2(e)
  float scale;
  uint64_t limit_ns;
  int* status;
};

// A work item: key tile kt of head bh and the query tiles qt0 .. qt0+n-1
// that see at least one of its keys.
struct Item {
  int bh, kt, qt0, n, key_limit;
};

__device__ __forceinline__ Item bwd_item(const Params& p, int t) {
  Item it;
  if (p.mask == kMaskCausal) {
    // key tiles with the most query tiles first (longest-processing-time order)
    it.kt = t / p.BH;
    it.bh = t % p.BH;
  } else {
    // the key tiles of one head back to back, so Q and dO stay hot in L2
    it.bh = t / p.num_kt;
    it.kt = t % p.num_kt;
  }
  int limit = p.n_k;
  if (p.mask == kMaskKeyPadding) {
    const int L = __ldg(p.key_lens + it.bh / p.H);
    limit = min(max(L, 0), p.n_k);
  }
  it.key_limit = limit;
  it.qt0 = 0;
  it.n = 0;
  if (it.kt * BN < limit) {
    if (p.mask == kMaskCausal) {
      // query i sees key j iff j <= i: tiles before kt see none of these keys
      it.qt0 = it.kt;
      it.n = max(p.num_qt - it.kt, 0);
    } else {
      it.n = p.num_qt;
    }
  }
  return it;
}

// Index of the next item of this CTA at or after `from` with work, or -1.
__device__ __forceinline__ int next_item(const Params& p, int from, Item& out) {
  for (int x = from; x < p.num_items; x += gridDim.x) {
    out = bwd_item(p, x);
    if (out.n > 0) return x;
  }
  return -1;
}

__device__ __forceinline__ void record_timeout(const Params& p, Smem& sm) {
  atomicCAS(p.status, kDevOk, kDevTimeout);
  *reinterpret_cast<volatile int*>(&sm.abort) = 1;
}

__device__ __forceinline__ void tma_reduce_add_3d(const CUtensorMap* map, uint32_t src, int x,
                                                  int y, int z) {
  asm volatile(
      "cp.reduce.async.bulk.tensor.3d.global.shared::cta.add.tile.bulk_group"
      " [%0, {%2, %3, %4}], [%1];" ::"l"(reinterpret_cast<uint64_t>(map)),
      "r"(src), "r"(x), "r"(y), "r"(z)
      : "memory");
}

// Contiguous global -> shared copy (size a multiple of 16, both addresses
// 16-byte aligned), completion counted on `bar` in bytes.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
      : "memory");
}

__device__ __forceinline__ float4 ld_shared_f4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr));
  return v;
}

// One row (128 bytes = eight 16-byte chunks) into a 128-byte swizzled tile:
// chunk g of row r lands at chunk position g ^ (r % 8).
__device__ __forceinline__ void st_row_sw128(uint32_t tile, int r, const uint32_t (&w)[32],
                                             int first_word) {
  const uint32_t base = tile + r * 128;
#pragma unroll
  for (int g = 0; g < 8; ++g)
    st_shared_v4(base + ((g ^ (r & 7)) << 4), w[first_word + 4 * g], w[first_word + 4 * g + 1],
                 w[first_word + 4 * g + 2], w[first_word + 4 * g + 3]);
}

__global__ void __launch_bounds__(NUM_THREADS, 1)
    attn_bwd_tc_kernel(const __grid_constant__ CUtensorMap tmq,
                       const __grid_constant__ CUtensorMap tmk,
                       const __grid_constant__ CUtensorMap tmv,
                       const __grid_constant__ CUtensorMap tmdo,
                       const __grid_constant__ CUtensorMap tmdk,
                       const __grid_constant__ CUtensorMap tmdv,
                       const __grid_constant__ CUtensorMap tmdq, const Params p) {
  extern __shared__ uint8_t smem_raw[];
  Smem& sm = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                      ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const volatile int* abort = &sm.abort;

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&sm.kv_full[i]), 1);
      mbar_init(smem_u32(&sm.kv_empty[i]), 1);
      mbar_init(smem_u32(&sm.q_full[i]), 1);
      mbar_init(smem_u32(&sm.q_empty[i]), 1);
    }
    mbar_init(smem_u32(&sm.s_full), 1);
    mbar_init(smem_u32(&sm.s_free), 256);
    mbar_init(smem_u32(&sm.dp_full), 1);
    mbar_init(smem_u32(&sm.dp_free), 256);
    mbar_init(smem_u32(&sm.p_full), 256);
    mbar_init(smem_u32(&sm.p_free), 1);
    mbar_init(smem_u32(&sm.ds_full), 256);
    mbar_init(smem_u32(&sm.ds_free), 1);
    mbar_init(smem_u32(&sm.dq_full), 1);
    mbar_init(smem_u32(&sm.dq_free), 128);
    mbar_init(smem_u32(&sm.dkv_full), 1);
    mbar_init(smem_u32(&sm.dkv_free), 128);
    mbar_init(smem_u32(&sm.drain), 1);
    sm.abort = 0;
    fence_mbar_init();
  }
  if (warp == LOAD_WARP && lane == 0) {
    prefetch_tmap(&tmq);
    prefetch_tmap(&tmk);
    prefetch_tmap(&tmv);
    prefetch_tmap(&tmdo);
    prefetch_tmap(&tmdk);
    prefetch_tmap(&tmdv);
    prefetch_tmap(&tmdq);
  }
  if (warp == MMA_WARP) {
    tmem_alloc(smem_u32(&sm.tmem_base), TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;

  if (warp == LOAD_WARP) {
    // -------------------------------------------------------------- producer
    if (lane == 0) {
      uint32_t it = 0, t = 0;
      bool ok = true;
      Item item;
      for (int x = next_item(p, blockIdx.x, item); x >= 0 && ok;
           x = next_item(p, x + gridDim.x, item), ++it) {
        const uint32_t slot = it & 1;
        ok = mbar_wait(smem_u32(&sm.kv_empty[slot]), ((it >> 1) & 1) ^ 1, p.limit_ns, abort);
        if (!ok) break;
        const uint32_t kvb = smem_u32(&sm.kv_full[slot]);
        mbar_arrive_expect_tx(kvb, 2 * TILE_BYTES);
        tma_load_3d(smem_u32(sm.k[slot]), &tmk, kvb, 0, item.kt * BN, item.bh);
        tma_load_3d(smem_u32(sm.v[slot]), &tmv, kvb, 0, item.kt * BN, item.bh);
        for (int i = 0; i < item.n && ok; ++i, ++t) {
          const uint32_t st = t & 1;
          ok = mbar_wait(smem_u32(&sm.q_empty[st]), ((t >> 1) & 1) ^ 1, p.limit_ns, abort);
          if (!ok) break;
          const int qt = item.qt0 + i;
          const uint32_t qb = smem_u32(&sm.q_full[st]);
          mbar_arrive_expect_tx(qb, 2 * TILE_BYTES + 2 * BM * 4);
          tma_load_3d(smem_u32(sm.q[st]), &tmq, qb, 0, qt * BM, item.bh);
          tma_load_3d(smem_u32(sm.dout[st]), &tmdo, qb, 0, qt * BM, item.bh);
          const size_t off = static_cast<size_t>(item.bh) * p.nq_pad + qt * BM;
          bulk_load(smem_u32(sm.nlse2[st]), p.nlse2 + off, BM * 4, qb);
          bulk_load(smem_u32(sm.nd[st]), p.nd + off, BM * 4, qb);
        }
      }
      if (!ok) {
        record_timeout(p, sm);
        // the copies already issued land before the shared memory goes away
        const int never = 0;
        for (uint32_t i = 0; i < 2; ++i) {
          const uint32_t kv_uses = it / 2 + (i < it % 2 ? 1u : 0u);
          if (kv_uses > 0)
            mbar_wait(smem_u32(&sm.kv_full[i]), (kv_uses - 1) & 1, p.limit_ns, &never);
          const uint32_t q_uses = t / 2 + (i < t % 2 ? 1u : 0u);
          if (q_uses > 0) mbar_wait(smem_u32(&sm.q_full[i]), (q_uses - 1) & 1, p.limit_ns, &never);
        }
      }
    }
  } else if (warp == MMA_WARP) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs the control flow; one elected lane issues.
    constexpr uint32_t IDESC_SQ = idesc_bf16_f32(BN, BM, false, false);  // S^T, dP^T
    constexpr uint32_t IDESC_KV = idesc_bf16_f32(BN, D, false, true);    // dV, dK
    constexpr uint32_t IDESC_DQ = idesc_bf16_f32(BM, D, true, true);     // dQ
    constexpr uint32_t T16 = TILE_BYTES >> 4;                            // a tile in desc units
    // K-major operands (rows x 64 bf16, 8-row groups 1024 B apart; a K step
    // of 16 elements is +32 B = +2 inside the swizzle row).
    const uint64_t kK = sdesc_sw128(smem_u32(sm.k[0]), 16, 1024);
    const uint64_t kV = sdesc_sw128(smem_u32(sm.v[0]), 16, 1024);
    const uint64_t kQ = sdesc_sw128(smem_u32(sm.q[0]), 16, 1024);
    const uint64_t kDO = sdesc_sw128(smem_u32(sm.dout[0]), 16, 1024);
    // P^T and dS^T as K-major A operands (M = keys, K = queries): a K step
    // inside a 64-query column block is +2, the second block is +16 KB.
    const uint64_t kPT = sdesc_sw128(smem_u32(sm.pt[0]), 16, 1024);
    const uint64_t kDST = sdesc_sw128(smem_u32(sm.dst[0]), 16, 1024);
    // MN-major B operands (K = the rows of the tile, N = the 64 columns): a K
    // step of 16 rows is +2048 B = +128; 8-row groups 1024 B apart (SBO); N
    // is one swizzle atom, LBO unused (set to 1024).
    const uint64_t nQ = sdesc_sw128(smem_u32(sm.q[0]), 1024, 1024);
    const uint64_t nDO = sdesc_sw128(smem_u32(sm.dout[0]), 1024, 1024);
    const uint64_t nK = sdesc_sw128(smem_u32(sm.k[0]), 1024, 1024);
    // dS as the MN-major A operand of dQ (M = queries across the two column
    // blocks, 16 KB apart = LBO; K = keys, 16 rows per step = +128).
    const uint64_t nDS = sdesc_sw128(smem_u32(sm.dst[0]), TILE_BYTES, 1024);

    const bool leader = elect_one();
    bool ok = true;
    auto wait = [&](uint64_t* bar, uint32_t parity) {
      if (ok) ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(bar), parity, p.limit_ns, abort));
      return ok;
    };
    auto issue_s = [&](uint32_t slot, uint32_t st) {  // S^T = K Q^T
      if (leader) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          mma_ss(tmem + COL_S, kK + slot * T16 + 2 * kk, kQ + st * T16 + 2 * kk, IDESC_SQ,
                 kk > 0 ? 1u : 0u);
        tc_commit(smem_u32(&sm.s_full));
      }
      __syncwarp();
    };
    auto issue_dp = [&](uint32_t slot, uint32_t st) {  // dP^T = V dO^T
      if (leader) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          mma_ss(tmem + COL_DP, kV + slot * T16 + 2 * kk, kDO + st * T16 + 2 * kk, IDESC_SQ,
                 kk > 0 ? 1u : 0u);
        tc_commit(smem_u32(&sm.dp_full));
      }
      __syncwarp();
    };

    uint32_t it = 0, t = 0;
    Item cur;
    int cx = next_item(p, blockIdx.x, cur);
    int ci = 0;  // index of tile t inside its item
    if (cx >= 0 && wait(&sm.kv_full[0], 0) && wait(&sm.q_full[0], 0)) {
      tc_fence_after();
      issue_s(0, 0);
      issue_dp(0, 0);
      while (ok) {
        const uint32_t slot = it & 1, st = t & 1;
        // dV += P^T dO (an item's first product overwrites dV, so the
        // epilogue must have read the previous item's dK and dV)
        if (ci == 0 && !wait(&sm.dkv_free, (it & 1) ^ 1)) break;
        if (!wait(&sm.p_full, t & 1)) break;
        tc_fence_after();
        if (leader) {
#pragma unroll
          for (int kk = 0; kk < BM / 16; ++kk)
            mma_ss(tmem + COL_DV, kPT + (kk >> 2) * T16 + 2 * (kk & 3), nDO + st * T16 + 128 * kk,
                   IDESC_KV, (ci > 0 || kk > 0) ? 1u : 0u);
          tc_commit(smem_u32(&sm.p_free));
        }
        __syncwarp();
        // the next tile pair's score products
        Item nx = cur;
        int nxx = cx, ni = ci + 1;
        uint32_t nit = it;
        if (ni >= cur.n) {
          nxx = next_item(p, cx + gridDim.x, nx);
          ni = 0;
          nit = it + 1;
        }
        const bool has_next = nxx >= 0;
        const uint32_t nslot = nit & 1, nst = (t + 1) & 1;
        if (has_next) {
          if (ni == 0 && !wait(&sm.kv_full[nslot], (nit >> 1) & 1)) break;
          if (!wait(&sm.q_full[nst], ((t + 1) >> 1) & 1)) break;
          if (!wait(&sm.s_free, t & 1)) break;
          tc_fence_after();
          issue_s(nslot, nst);
        }
        if (!wait(&sm.ds_full, t & 1)) break;
        tc_fence_after();
        if (has_next) {
          if (!wait(&sm.dp_free, t & 1)) break;
          tc_fence_after();
          issue_dp(nslot, nst);
        }
        // dK += dS^T Q
        if (leader) {
#pragma unroll
          for (int kk = 0; kk < BM / 16; ++kk)
            mma_ss(tmem + COL_DK, kDST + (kk >> 2) * T16 + 2 * (kk & 3), nQ + st * T16 + 128 * kk,
                   IDESC_KV, (ci > 0 || kk > 0) ? 1u : 0u);
        }
        __syncwarp();
        // dQ = dS K (the epilogue must have read the previous tile's dQ)
        if (!wait(&sm.dq_free, (t & 1) ^ 1)) break;
        tc_fence_after();
        if (leader) {
#pragma unroll
          for (int kk = 0; kk < BN / 16; ++kk)
            mma_ss(tmem + COL_DQ, nDS + 128 * kk, nK + slot * T16 + 128 * kk, IDESC_DQ,
                   kk > 0 ? 1u : 0u);
          tc_commit(smem_u32(&sm.dq_full));
          tc_commit(smem_u32(&sm.ds_free));
          tc_commit(smem_u32(&sm.q_empty[st]));
          if (ci == cur.n - 1) {
            tc_commit(smem_u32(&sm.kv_empty[slot]));
            tc_commit(smem_u32(&sm.dkv_full));
          }
        }
        __syncwarp();
        if (!has_next) break;
        cur = nx;
        cx = nxx;
        ci = ni;
        it = nit;
        ++t;
      }
    }
    if (!ok && leader) record_timeout(p, sm);
    // every MMA issued completes before tensor memory is freed
    if (leader) tc_commit(smem_u32(&sm.drain));
    __syncwarp();
    const int never = 0;
    mbar_wait(smem_u32(&sm.drain), 0, p.limit_ns, &never);
  } else if (warp >= EPI_WARP0) {
    // -------------------------------------------------------------- epilogue
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;  // tensor-memory lane = row of the tile
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const bool leader = quarter == 0 && lane == 0;
    const uint32_t stage = smem_u32(sm.stage);
    bool ok = true;
    auto wait = [&](uint64_t* bar, uint32_t parity) {
      if (ok) ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(bar), parity, p.limit_ns, abort));
      return ok;
    };
    // The staging buffer is free once the previous bulk copy has read it.
    auto stage_acquire = [&]() {
      if (leader) bulk_wait_read_all();
      named_bar_sync(EPI_BAR, 128);
    };
    auto stage_release = [&]() {
      fence_proxy_async_smem();
      named_bar_sync(EPI_BAR, 128);
    };
    uint32_t it = 0, t = 0;
    for (int x = blockIdx.x; x < p.num_items && ok; x += gridDim.x) {
      const Item item = bwd_item(p, x);
      uint32_t w[32];
      if (item.n == 0) {
        // no query sees these keys: dK = dV = 0
#pragma unroll
        for (int i = 0; i < 32; ++i) w[i] = 0u;
        stage_acquire();
        st_row_sw128(stage, r, w, 0);
        stage_release();
        if (leader) {
          tma_store_3d(&tmdk, stage, 0, item.kt * BN, item.bh);
          tma_store_3d(&tmdv, stage, 0, item.kt * BN, item.bh);
          bulk_commit_group();
        }
        continue;
      }
      for (int i = 0; i < item.n; ++i, ++t) {
        if (!wait(&sm.dq_full, t & 1)) break;
        tc_fence_after();
        uint32_t a[32], b[32];
        tmem_ld32(tmem + lane_off + COL_DQ, a);
        tmem_ld32(tmem + lane_off + COL_DQ + 32, b);
        tmem_ld_wait(a);
        reg_fence(b);
        tc_fence_before();
        mbar_arrive(smem_u32(&sm.dq_free));
        const int qt = item.qt0 + i;
        // two fp32 boxes of 32 columns (128 bytes a row), each added into
        // the accumulator by one TMA reduce; rows past n_q are not touched
        stage_acquire();
        st_row_sw128(stage, r, a, 0);
        stage_release();
        if (leader) {
          tma_reduce_add_3d(&tmdq, stage, 0, qt * BM, item.bh);
          bulk_commit_group();
        }
        stage_acquire();
        st_row_sw128(stage, r, b, 0);
        stage_release();
        if (leader) {
          tma_reduce_add_3d(&tmdq, stage, 32, qt * BM, item.bh);
          bulk_commit_group();
        }
      }
      if (!ok || !wait(&sm.dkv_full, it & 1)) break;
      tc_fence_after();
      // dV, then dK (times the scale), each through the staging buffer; the
      // accumulators are released once both are in registers
#pragma unroll 1
      for (int which = 0; which < 2; ++which) {
        uint32_t a[32], b[32], w[32];
        const uint32_t col = which == 0 ? COL_DV : COL_DK;
        const float sc = which == 0 ? 1.f : p.scale;
        tmem_ld32(tmem + lane_off + col, a);
        tmem_ld32(tmem + lane_off + col + 32, b);
        tmem_ld_wait(a);
        reg_fence(b);
        if (which == 1) {
          tc_fence_before();
          mbar_arrive(smem_u32(&sm.dkv_free));
        }
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          w[i] = pack_bf16x2(__uint_as_float(a[2 * i]) * sc, __uint_as_float(a[2 * i + 1]) * sc);
          w[16 + i] =
              pack_bf16x2(__uint_as_float(b[2 * i]) * sc, __uint_as_float(b[2 * i + 1]) * sc);
        }
        stage_acquire();
        st_row_sw128(stage, r, w, 0);
        stage_release();
        if (leader) {
          tma_store_3d(which == 0 ? &tmdv : &tmdk, stage, 0, item.kt * BN, item.bh);
          bulk_commit_group();
        }
      }
      ++it;
    }
    if (leader) bulk_wait_all();
    if (!ok) record_timeout(p, sm);
  } else {
    // ------------------------------------------------------- elementwise part
    const int quarter = warp & 3;
    const int half = warp >> 2;            // query columns 64*half .. 64*half+63
    const int r = quarter * 32 + lane;      // key row of the tile
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t tS = tmem + lane_off + COL_S + 64 * half;
    const uint32_t tDP = tmem + lane_off + COL_DP + 64 * half;
    const uint32_t pt_tile = smem_u32(sm.pt[half]);
    const uint32_t ds_tile = smem_u32(sm.dst[half]);
    const float c = p.scale_log2;
    bool ok = true;
    auto wait = [&](uint64_t* bar, uint32_t parity) {
      if (ok) ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(bar), parity, p.limit_ns, abort));
      return ok;
    };
    uint32_t t = 0;
    Item item;
    for (int x = next_item(p, blockIdx.x, item); x >= 0 && ok;
         x = next_item(p, x + gridDim.x, item)) {
      const int j = item.kt * BN + r;  // this thread's key
      const bool row_valid = j < item.key_limit;
      for (int i = 0; i < item.n; ++i, ++t) {
        const uint32_t st = t & 1;
        const int qt = item.qt0 + i;
        // leading columns whose query precedes this key (causal diagonal
        // tile), or all of them for a key past the sequence
        int lim = 0;
        if (!row_valid) {
          lim = 64;
        } else if (p.mask == kMaskCausal && qt == item.kt) {
          lim = min(max(r - 64 * half, 0), 64);
        }
        if (!wait(&sm.q_full[st], (t >> 1) & 1)) break;
        if (!wait(&sm.s_full, t & 1)) break;
        tc_fence_after();
        uint32_t s0[32], s1[32];
        tmem_ld32(tS, s0);
        tmem_ld32(tS + 32, s1);
        tmem_ld_wait(s0);
        reg_fence(s1);
        tc_fence_before();
        mbar_arrive(smem_u32(&sm.s_free));

        // P = 2^(S * scale * log2(e) - LSE * log2(e)), zero where forbidden
        const uint32_t lse_addr = smem_u32(&sm.nlse2[st][64 * half]);
        float pf[64];
#pragma unroll
        for (int g = 0; g < 16; ++g) {
          const float4 nl = ld_shared_f4(lse_addr + 16 * g);
          const uint32_t* src = g < 8 ? s0 + 4 * g : s1 + 4 * (g - 8);
          float x0, x1, x2, x3;
          fma2(x0, x1, __uint_as_float(src[0]), __uint_as_float(src[1]), c, c, nl.x, nl.y);
          fma2(x2, x3, __uint_as_float(src[2]), __uint_as_float(src[3]), c, c, nl.z, nl.w);
          const int c0 = 4 * g;
          pf[c0 + 0] = c0 + 0 < lim ? 0.f : ex2(x0);
          pf[c0 + 1] = c0 + 1 < lim ? 0.f : ex2(x1);
          pf[c0 + 2] = c0 + 2 < lim ? 0.f : ex2(x2);
          pf[c0 + 3] = c0 + 3 < lim ? 0.f : ex2(x3);
        }
        uint32_t w[32];
#pragma unroll
        for (int i2 = 0; i2 < 32; ++i2) w[i2] = pack_bf16x2(pf[2 * i2], pf[2 * i2 + 1]);
        // P^T of the previous tile pair has been read by its dV product
        if (!wait(&sm.p_free, (t & 1) ^ 1)) break;
        st_row_sw128(pt_tile, r, w, 0);
        fence_proxy_async_smem();
        mbar_arrive(smem_u32(&sm.p_full));

        // dS = P * (dP - D), stored 32 columns at a time once dS^T of the
        // previous tile pair has been read by its dK and dQ products
        if (!wait(&sm.dp_full, t & 1)) break;
        if (!wait(&sm.ds_free, (t & 1) ^ 1)) break;
        tc_fence_after();
        const uint32_t nd_addr = smem_u32(&sm.nd[st][64 * half]);
        const uint32_t ds_row = ds_tile + r * 128;
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
          uint32_t dp[32];
          tmem_ld32(tDP + 32 * h2, dp);
          tmem_ld_wait(dp);
          if (h2 == 1) {
            tc_fence_before();
            mbar_arrive(smem_u32(&sm.dp_free));
          }
#pragma unroll
          for (int g = 0; g < 4; ++g) {  // 8 columns = one 16-byte chunk
            uint32_t e[4];
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
              const int cc = 8 * g + 4 * hh;  // column inside the chunk of 32
              const float4 nd = ld_shared_f4(nd_addr + 128 * h2 + 4 * cc);
              const int c0 = 32 * h2 + cc;
              float d0, d1, d2, d3;
              add2(d0, d1, __uint_as_float(dp[cc]), __uint_as_float(dp[cc + 1]), nd.x, nd.y);
              add2(d2, d3, __uint_as_float(dp[cc + 2]), __uint_as_float(dp[cc + 3]), nd.z, nd.w);
              float e0, e1, e2, e3;
              fma2(e0, e1, pf[c0], pf[c0 + 1], d0, d1, 0.f, 0.f);
              fma2(e2, e3, pf[c0 + 2], pf[c0 + 3], d2, d3, 0.f, 0.f);
              e[2 * hh] = pack_bf16x2(e0, e1);
              e[2 * hh + 1] = pack_bf16x2(e2, e3);
            }
            const int chunk = 4 * h2 + g;
            st_shared_v4(ds_row + ((chunk ^ (r & 7)) << 4), e[0], e[1], e[2], e[3]);
          }
        }
        fence_proxy_async_smem();
        mbar_arrive(smem_u32(&sm.ds_full));
      }
    }
    if (!ok) record_timeout(p, sm);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == MMA_WARP) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

// Per query row (8 threads a row): -D = -sum_c dO_c O_c, -LSE * log2(e), and
// the dQ accumulator row set to zero.  Rows n_q .. nq_pad-1 of each head get
// zeros (their Q and dO rows are zero-filled by the tile loads).
__global__ void __launch_bounds__(256)
    attn_bwd_pre_kernel(const __nv_bfloat16* __restrict__ o, const __nv_bfloat16* __restrict__ dout,
                        const float* __restrict__ lse, float* __restrict__ nlse2,
                        float* __restrict__ nd, float* __restrict__ dq_acc, int n_q, int nq_pad,
                        long long rows) {
  const long long row = static_cast<long long>(blockIdx.x) * 32 + (threadIdx.x >> 3);
  const int sub = threadIdx.x & 7;
  const bool in = row < rows;
  const long long bh = in ? row / nq_pad : 0;
  const int i = in ? static_cast<int>(row - bh * nq_pad) : 0;
  const bool valid = in && i < n_q;
  const size_t src = (static_cast<size_t>(bh) * n_q + i) * D + sub * 8;
  float acc = 0.f;
  if (valid) {
    const uint4 a = *reinterpret_cast<const uint4*>(dout + src);
    const uint4 b = *reinterpret_cast<const uint4*>(o + src);
    const __nv_bfloat162* a2 = reinterpret_cast<const __nv_bfloat162*>(&a);
    const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&b);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 x = __bfloat1622float2(a2[e]);
      const float2 y = __bfloat1622float2(b2[e]);
      acc = fmaf(x.x, y.x, acc);
      acc = fmaf(x.y, y.y, acc);
    }
    float4* z = reinterpret_cast<float4*>(dq_acc + src);
    z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
    z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  acc += __shfl_xor_sync(0xffffffffu, acc, 4);
  acc += __shfl_xor_sync(0xffffffffu, acc, 2);
  acc += __shfl_xor_sync(0xffffffffu, acc, 1);
  if (in && sub == 0) {
    nd[row] = valid ? -acc : 0.f;
    nlse2[row] = valid ? -lse[static_cast<size_t>(bh) * n_q + i] * LOG2E : 0.f;
  }
}

// dQ = scale * accumulator, rounded to bf16; 8 elements a thread.
__global__ void __launch_bounds__(256)
    attn_bwd_dq_kernel(const float* __restrict__ dq_acc, __nv_bfloat16* __restrict__ dq,
                       float scale, long long n8) {
  const long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= n8) return;
  const float4 a = reinterpret_cast<const float4*>(dq_acc)[2 * i];
  const float4 b = reinterpret_cast<const float4*>(dq_acc)[2 * i + 1];
  uint4 out;
  out.x = pack_bf16x2(a.x * scale, a.y * scale);
  out.y = pack_bf16x2(a.z * scale, a.w * scale);
  out.z = pack_bf16x2(b.x * scale, b.y * scale);
  out.w = pack_bf16x2(b.z * scale, b.w * scale);
  reinterpret_cast<uint4*>(dq)[i] = out;
}

}  // namespace

BwdLayout bwd_layout(int B, int H, int n_q) {
  BwdLayout l;
  const size_t bh = static_cast<size_t>(B) * H;
  l.nq_pad = (n_q + BM - 1) / BM * BM;
  l.nlse2_off = 0;
  l.nd_off = bh * l.nq_pad * 4;
  l.dq_acc_off = 2 * bh * l.nq_pad * 4;
  l.bytes = l.dq_acc_off + bh * static_cast<size_t>(n_q) * D * 4;
  return l;
}

size_t bwd_tc_smem_bytes() { return sizeof(Smem) + 1024; }

cudaError_t launch_bwd(const BwdProblem& pb, const CUtensorMap* maps, void* workspace,
                       const LaunchCtx& ctx) {
  const BwdLayout lay = bwd_layout(pb.B, pb.H, pb.n_q);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  float* nlse2 = reinterpret_cast<float*>(ws + lay.nlse2_off);
  float* nd = reinterpret_cast<float*>(ws + lay.nd_off);
  float* dq_acc = reinterpret_cast<float*>(ws + lay.dq_acc_off);
  const long long bh = static_cast<long long>(pb.B) * pb.H;

  const long long rows = bh * lay.nq_pad;
  const long long pre_blocks = (rows + 31) / 32;
  attn_bwd_pre_kernel<<<static_cast<unsigned>(pre_blocks), 256, 0, ctx.stream>>>(
      static_cast<const __nv_bfloat16*>(pb.o), static_cast<const __nv_bfloat16*>(pb.dout), pb.lse,
      nlse2, nd, dq_acc, pb.n_q, static_cast<int>(lay.nq_pad), rows);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;

  Params p;
  p.nlse2 = nlse2;
  p.nd = nd;
  p.key_lens = pb.key_lens;
  p.H = pb.H;
  p.n_q = pb.n_q;
  p.n_k = pb.n_k;
  p.BH = static_cast<int>(bh);
  p.nq_pad = static_cast<int>(lay.nq_pad);
  p.mask = pb.mask;
  p.num_qt = (pb.n_q + BM - 1) / BM;
  p.num_kt = (pb.n_k + BN - 1) / BN;
  p.num_items = p.BH * p.num_kt;
  p.scale_log2 = pb.scale * LOG2E;
  p.scale = pb.scale;
  p.limit_ns = ctx.limit_ns;
  p.status = ctx.status;
  const size_t smem = bwd_tc_smem_bytes();
  err = cudaFuncSetAttribute(attn_bwd_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem));
  if (err != cudaSuccess) return err;
  const int grid = p.num_items < ctx.num_sms ? p.num_items : ctx.num_sms;
  attn_bwd_tc_kernel<<<grid, NUM_THREADS, smem, ctx.stream>>>(maps[0], maps[1], maps[2], maps[3],
                                                              maps[4], maps[5], maps[6], p);
  err = cudaGetLastError();
  if (err != cudaSuccess) return err;

  const long long n8 = bh * pb.n_q * (D / 8);
  attn_bwd_dq_kernel<<<static_cast<unsigned>((n8 + 255) / 256), 256, 0, ctx.stream>>>(
      dq_acc, static_cast<__nv_bfloat16*>(pb.dq), pb.scale, n8);
  return cudaGetLastError();
}

}  // namespace attn
