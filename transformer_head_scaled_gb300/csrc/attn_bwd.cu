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
//   1. attn_bwd_pre_kernel: per query row, the two per-query constants the
//      elementwise steps need, b_i = -LSE_i / scale and -D_i, each split into
//      three bf16 parts (hi + mid + lo) and written as [128 x 16] bf16 tiles;
//      and the row of the fp32 dQ accumulator set to zero.
//   2. attn_bwd_tc_kernel: one persistent CTA per SM walks work items = one
//      128-key tile of one (b, h); for each 128-query tile that the mask lets
//      see those keys it runs the tensor-core products of that tile pair and
//      accumulates dK and dV in tensor memory; dQ of the tile pair is added
//      into the fp32 accumulator in global memory with TMA reduces.
//   3. attn_bwd_dq_kernel: dQ = scale * accumulator, rounded to bf16.
//
// The per-query constants ride on the tensor cores: one extra K=16 step
// against an all-ones operand adds b_i to every score of column i and -D_i to
// every dP of column i,
//   S'^T = K Q^T + 1 b^T,   dP'^T = V dO^T + 1 (-D)^T,
// so that the elementwise work per element is P = 2^(scale*log2(e) * S') and
// dS = P * dP' (the three bf16 parts keep b and D to about 2^-24 relative).
//
// Kernel 2 (448 threads):
//   warps 0-7   elementwise: warp w owns tensor-memory lanes 32*(w%4).. (=
//               keys) and query columns 64*(w/4)..+63; it turns S'^T into P^T
//               (bf16, written to tensor memory) and dP'^T into dS^T (bf16,
//               written to shared memory in the 128-byte swizzled layout, two
//               buffers so that tile t+1's dS^T is written while dK(t) and
//               dQ(t) still read tile t's);
//   warps 8-11  epilogue, two groups of two warps (query or key rows 0-63 and
//               64-127), each with its own 8 KB staging buffer: dQ of each tile
//               pair (tensor memory -> swizzled fp32 staging -> TMA reduce-add
//               into the fp32 accumulator in global memory), dK and dV of each
//               item (-> bf16 -> TMA store);
//   warp  12    TMA producer: K per item (2 slots), V per item (1 slot: its
//               only reader, dP, is done with it a tile pair before the next
//               item needs it); Q and its constant tile (3 stages) and dO (2
//               stages) per query tile;
//   warp  13    tensor-memory owner and MMA issuer.
// Tensor memory (512 columns, w = max(d, 32) for head size d in {16, 32,
// 64}): S'^T [0,128)  dP'^T [128,256)  dV, dK, dQ w columns each from 256,
// then P^T (64 columns of bf16 pairs); at d = 64 dV [256,320) dK [320,384)
// dQ [384,448) P^T [448,512).  Keys are the 128 lanes of all but dQ, whose
// lanes are queries.  Q, K, V, dO tiles are [128 x d] in the swizzle of their
// 2d-byte rows; dS^T is [128 x 128] at every d.
// Products per tile pair t (all 128-row M; * = from tensor memory):
//   S'^T = K Q^T (+1 b^T)    dP'^T = V dO^T (+1 (-D)^T)    dV += P^T* dO
//   dK += dS^T Q             dQ = dS K
// issued in the order S'(t+1), dV(t), dP'(t+1), dK(t), dQ(t), so that the
// elementwise warps start on tile t+1 while the tensor pipe finishes the
// gradient products of tile t.  Every wait is bounded; on timeout the kernel
// records kDevTimeout, all roles drain and the CTA returns.
#include <cuda_bf16.h>

#include "attn_internal.cuh"
#include "ptx.cuh"

namespace attn {
namespace {

using namespace ptx;

constexpr int BM = 128;  // queries per query tile
constexpr int BN = 128;  // keys per key tile (= tensor-memory lanes)
constexpr uint32_t DS_BLOCK = 128 * 64 * 2;  // a [128 x 64] bf16 block of dS^T: 16 KB
// Q (and its constant tile) ring: Q is last read by dK, late in a tile pair,
// so three stages let the next tile's loads start two tile pairs ahead.  dO
// is last read by dV, early in a tile pair: two stages suffice.
constexpr int QSTAGES = 3;
constexpr int OSTAGES = 2;
constexpr int NUM_THREADS = 448;
constexpr int EPI_WARP0 = 8;
constexpr int LOAD_WARP = 12;
constexpr int MMA_WARP = 13;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t COL_S = 0, COL_DP = 128;
// The [128 x 16] bf16 constant tile of a query tile (K-major, no swizzle:
// 8-row x 16-byte core matrices, the second 8 columns 128 B after the first,
// 8-row groups 256 B apart).  Row i holds b_i in columns 0-2 (hi, mid, lo)
// and -D_i in columns 3-5; columns 6-15 are zero.
constexpr uint32_t CONST_TILE_BYTES = 128 * 16 * 2;
constexpr float LOG2E = 1.4426950408889634f;

static_assert(BM == BN, "the causal tile range assumes square tiles");

constexpr uint32_t STAGE_BYTES = 64 * 128;  // an epilogue staging buffer: 64 rows x 128 bytes
constexpr int EPI_BAR0 = 1;  // named barriers 1, 2: the two epilogue groups

// Shapes per head size d (16, 32, 64; d_k = d_v): Q, K, V and dO tiles of
// [128 x d] bf16 with rows of 2d bytes in the widest swizzle they fit; dV,
// dK and dQ accumulators of max(d, 32) tensor-memory columns (32-column
// loads never touch a neighbour); dQ added into the fp32 accumulator in boxes
// of min(d, 32) columns.  (d = 128 would need 704 tensor-memory columns.)
template <int D_>
struct BCfg {
  static constexpr uint32_t RB = D_ * 2;
  static constexpr uint32_t SWZ = RB == 128 ? 2u : (RB == 64 ? 4u : 6u);
  static constexpr uint32_t TILE = 128 * D_ * 2;
  static constexpr uint32_t OW = D_ < 32 ? 32 : D_;
  static constexpr uint32_t COL_DV = 256, COL_DK = 256 + OW, COL_DQ = 256 + 2 * OW,
                            COL_PT = 256 + 3 * OW;
  static constexpr uint32_t QRB = (D_ < 32 ? D_ : 32) * 4;  // row bytes of a dQ box
  static_assert(COL_PT + 64 <= 512, "tensor memory");
};

template <int D_>
struct __align__(1024) Smem {
  using C = BCfg<D_>;
  uint8_t k[2][C::TILE];
  uint8_t v[C::TILE];
  uint8_t q[QSTAGES][C::TILE];
  uint8_t dout[OSTAGES][C::TILE];
  // dS^T as [128 keys x 128 queries] bf16, two buffers (tile pairs t even /
  // odd), each two 64-query column blocks of [128 x 64] in the 128-byte
  // swizzled layout.
  uint8_t dst[2][2][DS_BLOCK];
  // epilogue staging, one 64-row buffer per epilogue group: a fp32 box of
  // dQ, or dV / dK in bf16, swizzled as the tensor map it is copied with
  uint8_t stage[2][STAGE_BYTES];
  uint8_t cst[QSTAGES][CONST_TILE_BYTES];  // the constant tile of each Q stage
  // Two 8 x 8 bf16 core matrices that select columns of the constant tile:
  // [0] rows (1,1,1,0,0,0,0,0) picks b, [1] rows (0,0,0,1,1,1,0,0) picks -D.
  uint8_t sel[2][512];
  uint64_t k_full[2], k_empty[2], v_full, v_empty;
  uint64_t q_full[QSTAGES], q_empty[QSTAGES];
  uint64_t o_full[OSTAGES], o_empty[OSTAGES];
  uint64_t s_full, s_free, dp_full, dp_free;
  uint64_t p_full, p_free, ds_full, ds_free[2];
  uint64_t dq_full, dq_free, dkv_full, dkv_free;
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};

struct Params {
  const uint8_t* cst;  // constant tiles [BH][num_qt][CONST_TILE_BYTES]
  const int* key_lens;
  int H, n_q, n_k, BH;
  int mask;
  int win_left, win_right;  // restricted attention: query i sees keys i - left .. i + right
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
    } else if (p.mask == kMaskBand) {
      // key j is seen by the queries j - right .. j + left
      const int j_lo = it.kt * BN, j_hi = min(j_lo + BN - 1, limit - 1);
      const int q_lo = max(j_lo - p.win_right, 0), q_hi = min(j_hi + p.win_left, p.n_q - 1);
      if (q_lo <= q_hi) {
        it.qt0 = q_lo / BM;
        it.n = q_hi / BM - it.qt0 + 1;
      }
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

template <class SmemT>
__device__ __forceinline__ void record_timeout(const Params& p, SmemT& sm) {
  atomicCAS(p.status, kDevOk, kDevTimeout);
  *reinterpret_cast<volatile int*>(&sm.abort) = 1;
}

// 3-D tiled reduce-add shared -> global (fp32 add, element type from the
// tensor map), tracked by the issuing thread's bulk groups.  Parts of the box
// outside the tensor are not touched.
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

// Shared-memory matrix descriptor without swizzle (K-major: 8-row x 16-byte
// core matrices; LBO = byte step between the two 8-column halves of K = 16,
// SBO = byte step between 8-row groups).  Same fields as the 128-byte swizzle
// descriptor with layout bits 61-63 = 0.
__device__ __forceinline__ uint64_t sdesc_plain(uint32_t smem_addr, uint32_t lbo_bytes,
                                                uint32_t sbo_bytes) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((smem_addr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>((lbo_bytes >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo_bytes >> 4) & 0x3FFFu) << 32;
  d |= 1ull << 46;
  return d;
}

// One row of RBYTES (128, 64 or 32) into a tile swizzled at that width:
// 16-byte chunk g of row r lands at chunk position g ^ ((r * RBYTES / 128) %
// (RBYTES / 16)), the layout a TMA copy with that swizzle reads and writes.
template <uint32_t RBYTES>
__device__ __forceinline__ void st_row_swz(uint32_t tile, int r, const uint32_t (&w)[32]) {
  const uint32_t base = tile + r * RBYTES;
  const uint32_t x = ((static_cast<uint32_t>(r) * RBYTES) >> 7) & (RBYTES / 16 - 1);
#pragma unroll
  for (uint32_t g = 0; g < RBYTES / 16; ++g)
    st_shared_v4(base + ((g ^ x) << 4), w[4 * g], w[4 * g + 1], w[4 * g + 2], w[4 * g + 3]);
}

// Shared-memory matrix descriptor (same fields as sdesc_sw128) with the
// layout code `swz` at bits 61-63.
__device__ __forceinline__ uint64_t sdesc_swz(uint32_t smem_addr, uint32_t lbo_bytes,
                                              uint32_t sbo_bytes, uint32_t swz) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((smem_addr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>((lbo_bytes >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo_bytes >> 4) & 0x3FFFu) << 32;
  d |= 1ull << 46;
  d |= static_cast<uint64_t>(swz) << 61;
  return d;
}

// BAND = restricted self-attention (its own instantiation, so that the
// window's two extra compares per score stay out of the other masks' code).
template <bool BAND, int D_>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    attn_bwd_tc_kernel(const __grid_constant__ CUtensorMap tmq,
                       const __grid_constant__ CUtensorMap tmk,
                       const __grid_constant__ CUtensorMap tmv,
                       const __grid_constant__ CUtensorMap tmdo,
                       const __grid_constant__ CUtensorMap tmdk,
                       const __grid_constant__ CUtensorMap tmdv,
                       const __grid_constant__ CUtensorMap tmdq, const Params p) {
  using C = BCfg<D_>;
  constexpr int D = D_;
  extern __shared__ uint8_t smem_raw[];
  Smem<D_>& sm = *reinterpret_cast<Smem<D_>*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const volatile int* abort = &sm.abort;

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&sm.k_full[i]), 1);
      mbar_init(smem_u32(&sm.k_empty[i]), 1);
    }
    mbar_init(smem_u32(&sm.v_full), 1);
    mbar_init(smem_u32(&sm.v_empty), 1);
    for (int i = 0; i < QSTAGES; ++i) {
      mbar_init(smem_u32(&sm.q_full[i]), 1);
      mbar_init(smem_u32(&sm.q_empty[i]), 1);
    }
    for (int i = 0; i < OSTAGES; ++i) {
      mbar_init(smem_u32(&sm.o_full[i]), 1);
      mbar_init(smem_u32(&sm.o_empty[i]), 1);
    }
    mbar_init(smem_u32(&sm.s_full), 1);
    mbar_init(smem_u32(&sm.s_free), 256);
    mbar_init(smem_u32(&sm.dp_full), 1);
    mbar_init(smem_u32(&sm.dp_free), 256);
    mbar_init(smem_u32(&sm.p_full), 256);
    mbar_init(smem_u32(&sm.p_free), 1);
    mbar_init(smem_u32(&sm.ds_full), 256);
    mbar_init(smem_u32(&sm.ds_free[0]), 1);
    mbar_init(smem_u32(&sm.ds_free[1]), 1);
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
  if (warp == 0) {
    // the selector operands of the constant products (bf16 1.0 = 0x3F80):
    // word w of a 16-byte row holds columns 2w, 2w+1
    const uint32_t wi = lane & 3;
    const uint32_t sb = wi == 0 ? 0x3F803F80u : (wi == 1 ? 0x00003F80u : 0u);
    const uint32_t sd = wi == 1 ? 0x3F800000u : (wi == 2 ? 0x3F803F80u : 0u);
    reinterpret_cast<uint32_t*>(sm.sel[0])[lane] = sb;
    reinterpret_cast<uint32_t*>(sm.sel[1])[lane] = sd;
    fence_proxy_async_smem();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  // Launched as a dependent of the preprocess kernel (which writes the
  // constant tiles and zeroes the dQ accumulator): everything above overlaps
  // its tail, nothing below runs before it has completed.
  grid_dependency_wait();

  if (warp == LOAD_WARP) {
    // -------------------------------------------------------------- producer
    if (lane == 0) {
      uint32_t it = 0, nv = 0, nq = 0, no = 0;  // K, V, Q and dO loads issued
      bool ok = true;
      Item item;
      for (int x = next_item(p, blockIdx.x, item); x >= 0 && ok;
           x = next_item(p, x + gridDim.x, item)) {
        const uint32_t slot = it & 1;
        ok = mbar_wait(smem_u32(&sm.k_empty[slot]), ((it >> 1) & 1) ^ 1, p.limit_ns, abort);
        if (!ok) break;
        mbar_arrive_expect_tx(smem_u32(&sm.k_full[slot]), C::TILE);
        tma_load_4d(smem_u32(sm.k[slot]), &tmk, smem_u32(&sm.k_full[slot]), 0, item.kt * BN,
                    item.bh % p.H, item.bh / p.H);
        ++it;
        for (int i = 0; i < item.n && ok; ++i) {
          const int qt = item.qt0 + i;
          const uint32_t st = nq % QSTAGES;
          ok = mbar_wait(smem_u32(&sm.q_empty[st]), ((nq / QSTAGES) & 1) ^ 1, p.limit_ns, abort);
          if (!ok) break;
          const uint32_t qb = smem_u32(&sm.q_full[st]);
          mbar_arrive_expect_tx(qb, C::TILE + CONST_TILE_BYTES);
          tma_load_4d(smem_u32(sm.q[st]), &tmq, qb, 0, qt * BM, item.bh % p.H, item.bh / p.H);
          const size_t tile = static_cast<size_t>(item.bh) * p.num_qt + qt;
          bulk_load(smem_u32(sm.cst[st]), p.cst + tile * CONST_TILE_BYTES, CONST_TILE_BYTES, qb);
          ++nq;
          if (i == 0) {
            // V of this item, once the previous item's last dP has read the slot
            ok = mbar_wait(smem_u32(&sm.v_empty), (nv & 1) ^ 1, p.limit_ns, abort);
            if (!ok) break;
            mbar_arrive_expect_tx(smem_u32(&sm.v_full), C::TILE);
            tma_load_4d(smem_u32(sm.v), &tmv, smem_u32(&sm.v_full), 0, item.kt * BN,
                        item.bh % p.H, item.bh / p.H);
            ++nv;
          }
          const uint32_t os = no % OSTAGES;
          ok = mbar_wait(smem_u32(&sm.o_empty[os]), ((no / OSTAGES) & 1) ^ 1, p.limit_ns, abort);
          if (!ok) break;
          const uint32_t ob = smem_u32(&sm.o_full[os]);
          mbar_arrive_expect_tx(ob, C::TILE);
          tma_load_4d(smem_u32(sm.dout[os]), &tmdo, ob, 0, qt * BM, item.bh % p.H,
                      item.bh / p.H);
          ++no;
        }
      }
      if (!ok) {
        record_timeout(p, sm);
        // the copies already issued land before the shared memory goes away:
        // wait (bounded, ignoring the abort flag) for the last phase armed on
        // every full barrier
        const int never = 0;
        auto drain = [&](uint64_t* full, uint32_t stages, uint32_t issued) {
          for (uint32_t i = 0; i < stages; ++i) {
            const uint32_t uses = issued / stages + (i < issued % stages ? 1u : 0u);
            if (uses > 0) mbar_wait(smem_u32(&full[i]), (uses - 1) & 1, p.limit_ns, &never);
          }
        };
        drain(sm.k_full, 2, it);
        drain(&sm.v_full, 1, nv);
        drain(sm.q_full, QSTAGES, nq);
        drain(sm.o_full, OSTAGES, no);
      }
    }
  } else if (warp == MMA_WARP) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs the control flow; one elected lane issues.
    constexpr uint32_t IDESC_SQ = idesc_bf16_f32(BN, BM, false, false);  // S^T, dP^T
    constexpr uint32_t IDESC_KV = idesc_bf16_f32(BN, D, false, true);    // dV (A in tensor memory), dK
    constexpr uint32_t IDESC_DQ = idesc_bf16_f32(BM, D, true, true);     // dQ
    constexpr uint32_t T16 = C::TILE >> 4;     // a [128 x d] tile in desc units
    constexpr uint32_t DS16 = DS_BLOCK >> 4;   // a dS^T column block in desc units
    constexpr uint32_t RB16 = C::RB;           // 16 rows of RB bytes in desc units
    // K-major operands (rows x d bf16, 8-row groups 8*RB bytes apart; a K
    // step of 16 elements is +32 B = +2 inside the swizzle row).
    const uint64_t kK = sdesc_swz(smem_u32(sm.k[0]), 16, 8 * C::RB, C::SWZ);
    const uint64_t kV = sdesc_swz(smem_u32(sm.v), 16, 8 * C::RB, C::SWZ);
    const uint64_t kQ = sdesc_swz(smem_u32(sm.q[0]), 16, 8 * C::RB, C::SWZ);
    const uint64_t kDO = sdesc_swz(smem_u32(sm.dout[0]), 16, 8 * C::RB, C::SWZ);
    // dS^T as the K-major A operand of dK (M = keys, K = queries): a K step
    // inside a 64-query column block is +2, the second block is +16 KB.
    const uint64_t kDST = sdesc_sw128(smem_u32(sm.dst[0][0]), 16, 1024);
    // MN-major B operands (K = the rows of the tile, N = the d columns): a K
    // step of 16 rows is 16*RB bytes (+RB16); 8-row groups 8*RB bytes apart
    // (SBO); N is one swizzle atom, LBO unused (set to 1024).
    const uint64_t nQ = sdesc_swz(smem_u32(sm.q[0]), 1024, 8 * C::RB, C::SWZ);
    const uint64_t nDO = sdesc_swz(smem_u32(sm.dout[0]), 1024, 8 * C::RB, C::SWZ);
    const uint64_t nK = sdesc_swz(smem_u32(sm.k[0]), 1024, 8 * C::RB, C::SWZ);
    // dS as the MN-major A operand of dQ (M = queries across the two column
    // blocks, 16 KB apart = LBO; K = keys, 16 rows per step = +128).
    const uint64_t nDS = sdesc_sw128(smem_u32(sm.dst[0][0]), DS_BLOCK, 1024);
    // The constant products: A = a selector (every core matrix of the 128 x 16
    // operand aliases the same 128 bytes: LBO = SBO = 0), B = the Q stage's
    // [128 queries x 16] constant tile.
    const uint64_t kSelB = sdesc_plain(smem_u32(sm.sel[0]), 0, 0);
    const uint64_t kSelD = sdesc_plain(smem_u32(sm.sel[1]), 0, 0);
    const uint64_t kCst = sdesc_plain(smem_u32(sm.cst[0]), 128, 256);
    constexpr uint32_t C16 = CONST_TILE_BYTES >> 4;

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
        mma_ss(tmem + COL_S, kSelB, kCst + st * C16, IDESC_SQ, 1u);  // + b_i
        tc_commit(smem_u32(&sm.s_full));
      }
      __syncwarp();
    };
    // dP^T = V dO^T; the last tile pair of an item releases the V slot
    auto issue_dp = [&](uint32_t qs, uint32_t os, bool last_of_item) {
      if (leader) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          mma_ss(tmem + COL_DP, kV + 2 * kk, kDO + os * T16 + 2 * kk, IDESC_SQ, kk > 0 ? 1u : 0u);
        mma_ss(tmem + COL_DP, kSelD, kCst + qs * C16, IDESC_SQ, 1u);  // - D_i
        tc_commit(smem_u32(&sm.dp_full));
        if (last_of_item) tc_commit(smem_u32(&sm.v_empty));
      }
      __syncwarp();
    };

    uint32_t it = 0, t = 0;
    Item cur;
    int cx = next_item(p, blockIdx.x, cur);
    int ci = 0;  // index of tile t inside its item
    if (cx >= 0 && wait(&sm.k_full[0], 0) && wait(&sm.q_full[0], 0) && wait(&sm.v_full, 0) &&
        wait(&sm.o_full[0], 0)) {
      tc_fence_after();
      issue_s(0, 0);
      issue_dp(0, 0, cur.n == 1);
      while (ok) {
        const uint32_t slot = it & 1, st = t % QSTAGES, os = t % OSTAGES;
        // the next tile pair (possibly of the next item)
        Item nx = cur;
        int nxx = cx, ni = ci + 1;
        uint32_t nit = it;
        if (ni >= cur.n) {
          nxx = next_item(p, cx + gridDim.x, nx);
          ni = 0;
          nit = it + 1;
        }
        const bool has_next = nxx >= 0;
        const uint32_t nslot = nit & 1, nst = (t + 1) % QSTAGES, nos = (t + 1) % OSTAGES;
        // its score product goes first, as soon as S'^T of this one is in the
        // elementwise warps' registers
        if (has_next) {
          if (ni == 0 && !wait(&sm.k_full[nslot], (nit >> 1) & 1)) break;
          if (!wait(&sm.q_full[nst], ((t + 1) / QSTAGES) & 1)) break;
          if (!wait(&sm.s_free, t & 1)) break;
          tc_fence_after();
          issue_s(nslot, nst);
        }
        // dV += P^T dO (an item's first product overwrites dV, so the
        // epilogue must have read the previous item's dK and dV)
        if (ci == 0 && !wait(&sm.dkv_free, (it & 1) ^ 1)) break;
        if (!wait(&sm.p_full, t & 1)) break;
        tc_fence_after();
        if (leader) {
#pragma unroll
          for (int kk = 0; kk < BM / 16; ++kk)
            mma_ts(tmem + C::COL_DV, tmem + C::COL_PT + 8 * kk, nDO + os * T16 + RB16 * kk, IDESC_KV,
                   (ci > 0 || kk > 0) ? 1u : 0u);
          tc_commit(smem_u32(&sm.p_free));
          tc_commit(smem_u32(&sm.o_empty[os]));  // the last product that reads this dO
        }
        __syncwarp();
        if (!wait(&sm.ds_full, t & 1)) break;
        tc_fence_after();
        if (has_next) {
          if (!wait(&sm.dp_free, t & 1)) break;
          if (ni == 0 && !wait(&sm.v_full, nit & 1)) break;
          if (!wait(&sm.o_full[nos], ((t + 1) / OSTAGES) & 1)) break;
          tc_fence_after();
          issue_dp(nst, nos, ni == nx.n - 1);
        }
        // dK += dS^T Q (the last product that reads this stage's Q)
        if (leader) {
#pragma unroll
          for (int kk = 0; kk < BM / 16; ++kk)
            mma_ss(tmem + C::COL_DK, kDST + (2 * (t & 1) + (kk >> 2)) * DS16 + 2 * (kk & 3),
                   nQ + st * T16 + RB16 * kk, IDESC_KV, (ci > 0 || kk > 0) ? 1u : 0u);
          tc_commit(smem_u32(&sm.q_empty[st]));
        }
        __syncwarp();
        // dQ = dS K (the epilogue must have read the previous tile's dQ)
        if (!wait(&sm.dq_free, (t & 1) ^ 1)) break;
        tc_fence_after();
        if (leader) {
#pragma unroll
          for (int kk = 0; kk < BN / 16; ++kk)
            mma_ss(tmem + C::COL_DQ, nDS + 2 * (t & 1) * DS16 + 128 * kk,
                   nK + slot * T16 + RB16 * kk, IDESC_DQ, kk > 0 ? 1u : 0u);
          tc_commit(smem_u32(&sm.dq_full));
          tc_commit(smem_u32(&sm.ds_free[t & 1]));
          if (ci == cur.n - 1) {
            tc_commit(smem_u32(&sm.k_empty[slot]));
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
    // group g = rows 64g .. 64g+63 (warps 8+2g, 9+2g), staging buffer g
    const int g = quarter >> 1;
    const int rg = r & 63;  // row inside the group's 64-row box
    const bool leader = (quarter & 1) == 0 && lane == 0;
    const uint32_t stage = smem_u32(sm.stage[g]);
    const uint32_t bar_id = EPI_BAR0 + g;
    bool ok = true;
    auto wait = [&](uint64_t* bar, uint32_t parity) {
      if (ok) ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(bar), parity, p.limit_ns, abort));
      return ok;
    };
    // The group's buffer is free once its previous bulk copy has read it;
    // after the rows are written, the copy may start.
    auto stage_acquire = [&]() {
      if (leader) bulk_wait_read_all();
      named_bar_sync(bar_id, 64);
    };
    auto stage_release = [&]() {
      fence_proxy_async_smem();
      named_bar_sync(bar_id, 64);
    };
    uint32_t it = 0, t = 0;
    for (int x = blockIdx.x; x < p.num_items && ok; x += gridDim.x) {
      const Item item = bwd_item(p, x);
      const int key_row0 = item.kt * BN + 64 * g;
      if (item.n == 0) {
        // no query sees these keys: dK = dV = 0
        uint32_t w[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) w[i] = 0u;
        stage_acquire();
        st_row_swz<C::RB>(stage, rg, w);
        stage_release();
        if (leader && key_row0 < p.n_k) {
          tma_store_4d(&tmdk, stage, 0, key_row0, item.bh % p.H, item.bh / p.H);
          tma_store_4d(&tmdv, stage, 0, key_row0, item.bh % p.H, item.bh / p.H);
          bulk_commit_group();
        }
        continue;
      }
      for (int i = 0; i < item.n; ++i, ++t) {
        if (!wait(&sm.dq_full, t & 1)) break;
        tc_fence_after();
        uint32_t a[32], b[32];
        tmem_ld32(tmem + lane_off + C::COL_DQ, a);
        if constexpr (D > 32) tmem_ld32(tmem + lane_off + C::COL_DQ + 32, b);
        tmem_ld_wait(a);
        if constexpr (D > 32) reg_fence(b);
        tc_fence_before();
        mbar_arrive(smem_u32(&sm.dq_free));
        // fp32 boxes of min(d, 32) columns x 64 rows per group, each added
        // into the accumulator by one TMA reduce; rows past n_q are not touched
        const int q_row0 = (item.qt0 + i) * BM + 64 * g;
        stage_acquire();
        st_row_swz<C::QRB>(stage, rg, a);
        stage_release();
        if (leader && q_row0 < p.n_q) {
          tma_reduce_add_3d(&tmdq, stage, 0, q_row0, item.bh);
          bulk_commit_group();
        }
        if constexpr (D > 32) {
          stage_acquire();
          st_row_swz<C::QRB>(stage, rg, b);
          stage_release();
          if (leader && q_row0 < p.n_q) {
            tma_reduce_add_3d(&tmdq, stage, 32, q_row0, item.bh);
            bulk_commit_group();
          }
        }
      }
      if (!ok || !wait(&sm.dkv_full, it & 1)) break;
      tc_fence_after();
      // dV, then dK (times the scale); the accumulators are released once
      // both are in registers
#pragma unroll 1
      for (int which = 0; which < 2; ++which) {
        uint32_t a[32], b[32], w[32];
        const uint32_t col = which == 0 ? C::COL_DV : C::COL_DK;
        const float sc = which == 0 ? 1.f : p.scale;
        tmem_ld32(tmem + lane_off + col, a);
        if constexpr (D > 32) tmem_ld32(tmem + lane_off + col + 32, b);
        tmem_ld_wait(a);
        if constexpr (D > 32) reg_fence(b);
        if (which == 1) {
          tc_fence_before();
          mbar_arrive(smem_u32(&sm.dkv_free));
        }
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          if (i < D / 2)
            w[i] = pack_bf16x2(__uint_as_float(a[2 * i]) * sc, __uint_as_float(a[2 * i + 1]) * sc);
          if constexpr (D > 32)
            w[16 + i] =
                pack_bf16x2(__uint_as_float(b[2 * i]) * sc, __uint_as_float(b[2 * i + 1]) * sc);
        }
        stage_acquire();
        st_row_swz<C::RB>(stage, rg, w);
        stage_release();
        if (leader && key_row0 < p.n_k) {
          tma_store_4d(which == 0 ? &tmdv : &tmdk, stage, 0, key_row0, item.bh % p.H,
                       item.bh / p.H);
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
    const uint32_t tPT = tmem + lane_off + C::COL_PT + 32 * half;
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
        const int qt = item.qt0 + i;
        // leading columns whose query precedes this key (causal diagonal
        // tile), or all of them for a key past the sequence; with the window,
        // the columns outside [lim, hi) (queries i with j < i - left or
        // j > i + right)
        int lim = 0, hi = 64;
        if (!row_valid) {
          lim = 64;
        } else if (p.mask == kMaskCausal && qt == item.kt) {
          lim = min(max(r - 64 * half, 0), 64);
        } else if (BAND) {
          const int qbase = qt * BM + 64 * half;
          lim = min(max(j - p.win_right - qbase, 0), 64);
          hi = min(max(j + p.win_left - qbase + 1, 0), 64);
        }
        if (!wait(&sm.s_full, t & 1)) break;
        tc_fence_after();
        uint32_t s0[32], s1[32];
        tmem_ld32(tS, s0);
        tmem_ld32(tS + 32, s1);
        tmem_ld_wait(s0);
        reg_fence(s1);
        tc_fence_before();
        mbar_arrive(smem_u32(&sm.s_free));

        // P = 2^(scale * log2(e) * S') (S' already holds -LSE/scale), zero
        // where forbidden
        float pf[64];
#pragma unroll
        for (int i2 = 0; i2 < 32; i2 += 2) {
          const uint32_t* src = i2 < 16 ? s0 + 2 * i2 : s1 + 2 * (i2 - 16);
          float x0, x1, x2, x3;
          fma2(x0, x1, __uint_as_float(src[0]), __uint_as_float(src[1]), c, c, 0.f, 0.f);
          fma2(x2, x3, __uint_as_float(src[2]), __uint_as_float(src[3]), c, c, 0.f, 0.f);
          const int c0 = 2 * i2;
          pf[c0 + 0] = (c0 + 0 < lim || (BAND && c0 + 0 >= hi)) ? 0.f : ex2(x0);
          pf[c0 + 1] = (c0 + 1 < lim || (BAND && c0 + 1 >= hi)) ? 0.f : ex2(x1);
          pf[c0 + 2] = (c0 + 2 < lim || (BAND && c0 + 2 >= hi)) ? 0.f : ex2(x2);
          pf[c0 + 3] = (c0 + 3 < lim || (BAND && c0 + 3 >= hi)) ? 0.f : ex2(x3);
        }
        uint32_t w[32];
#pragma unroll
        for (int i2 = 0; i2 < 32; ++i2) w[i2] = pack_bf16x2(pf[2 * i2], pf[2 * i2 + 1]);
        // P^T of the previous tile pair has been read by its dV product
        if (!wait(&sm.p_free, (t & 1) ^ 1)) break;
        tc_fence_after();
        tmem_st32(tPT, w);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(smem_u32(&sm.p_full));

        // dS = P * dP' (dP' already holds -D), computed into registers while
        // the previous tile pair's dK and dQ products still read dS^T
        if (!wait(&sm.dp_full, t & 1)) break;
        tc_fence_after();
        uint32_t e[32];  // dS as bf16 pairs, columns 2i, 2i+1
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
          for (int cc = 0; cc < 32; cc += 4) {
            const int c0 = 32 * h2 + cc;
            float e0, e1, e2, e3;
            fma2(e0, e1, pf[c0], pf[c0 + 1], __uint_as_float(dp[cc]), __uint_as_float(dp[cc + 1]),
                 0.f, 0.f);
            fma2(e2, e3, pf[c0 + 2], pf[c0 + 3], __uint_as_float(dp[cc + 2]),
                 __uint_as_float(dp[cc + 3]), 0.f, 0.f);
            e[c0 / 2] = pack_bf16x2(e0, e1);
            e[c0 / 2 + 1] = pack_bf16x2(e2, e3);
          }
        }
        // dS^T buffer t % 2 was last read by the products of tile pair t - 2
        if (!wait(&sm.ds_free[t & 1], ((t >> 1) & 1) ^ 1)) break;
        st_row_swz<128>(smem_u32(sm.dst[t & 1][half]), r, e);
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

// x as hi + mid + lo, three bf16 values (each the rounding of what the
// previous ones leave; together within about 2^-24 of x).
__device__ __forceinline__ uint2 split3_bf16(float x) {
  const __nv_bfloat16 hi = __float2bfloat16_rn(x);
  const float r1 = x - __bfloat162float(hi);
  const __nv_bfloat16 mid = __float2bfloat16_rn(r1);
  const float r2 = r1 - __bfloat162float(mid);
  const __nv_bfloat16 lo = __float2bfloat16_rn(r2);
  uint2 w;
  w.x = static_cast<uint32_t>(__bfloat16_as_ushort(hi)) |
        (static_cast<uint32_t>(__bfloat16_as_ushort(mid)) << 16);
  w.y = static_cast<uint32_t>(__bfloat16_as_ushort(lo));
  return w;
}

// Per query row (d/8 threads a row, 8 elements each): D = sum_c dO_c O_c, the constant tile's
// row for this query (b = -LSE/scale and -D, three bf16 parts each), and the
// dQ accumulator row set to zero.  Rows n_q .. of the last query tile get zero
// constants (their Q and dO rows are zero-filled by the tile loads, so every
// product they enter is zero).
template <int D>
__global__ void __launch_bounds__(256)
    attn_bwd_pre_kernel(const __nv_bfloat16* __restrict__ o, const __nv_bfloat16* __restrict__ dout,
                        const float* __restrict__ lse, uint8_t* __restrict__ cst,
                        float* __restrict__ dq_acc, int H, int n_q, int num_qt, float inv_scale,
                        long long rows, RowStrides so, RowStrides sdo) {
  // the main kernel may start launching now: it waits for this grid to
  // complete before it reads the constants or adds into dq_acc
  grid_launch_dependents();
  constexpr int TPR = D / 8;  // threads a row
  const long long row = static_cast<long long>(blockIdx.x) * (256 / TPR) + threadIdx.x / TPR;
  const int sub = threadIdx.x % TPR;
  const bool in = row < rows;
  const long long per_head = static_cast<long long>(num_qt) * BM;
  const long long bh = in ? row / per_head : 0;
  const int i = in ? static_cast<int>(row - bh * per_head) : 0;  // query index
  const bool valid = in && i < n_q;
  const size_t src = (static_cast<size_t>(bh) * n_q + i) * D + sub * 8;  // accumulator row
  const long long bb = bh / H, hh = bh % H;
  float acc = 0.f;
  if (valid) {
    const uint4 a =
        *reinterpret_cast<const uint4*>(dout + bb * sdo.b + hh * sdo.h + i * sdo.n + sub * 8);
    const uint4 b = *reinterpret_cast<const uint4*>(o + bb * so.b + hh * so.h + i * so.n + sub * 8);
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
#pragma unroll
  for (int m = TPR / 2; m > 0; m >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, m);
  if (in && sub < 2) {
    // sub 0: columns 0-7 of this query's row (b in 0-2, -D in 3-5); sub 1:
    // columns 8-15, zero
    const int qt = i / BM, n = i % BM;
    uint8_t* tile =
        cst + (static_cast<size_t>(bh) * num_qt + qt) * static_cast<size_t>(CONST_TILE_BYTES);
    uint4 w = make_uint4(0u, 0u, 0u, 0u);
    if (sub == 0 && valid) {
      const float l = lse[static_cast<size_t>(bh) * n_q + i];
      const float b = isfinite(l) ? -l * inv_scale : 0.f;  // -inf only for a row that sees no key
      const uint2 pb = split3_bf16(b);
      const uint2 pd = split3_bf16(-acc);
      w.x = pb.x;                         // b_hi, b_mid
      w.y = pb.y | (pd.x << 16);          // b_lo, -D_hi
      w.z = (pd.x >> 16) | (pd.y << 16);  // -D_mid, -D_lo
    }
    *reinterpret_cast<uint4*>(tile + (n & 7) * 16 + (n >> 3) * 256 + sub * 128) = w;
  }
}

// dQ = scale * accumulator, rounded to bf16, written through dq's strides;
// 8 elements a thread (d8 = d / 8 threads a row).
__global__ void __launch_bounds__(256)
    attn_bwd_dq_kernel(const float* __restrict__ dq_acc, __nv_bfloat16* __restrict__ dq,
                       float scale, long long n8, int d8, int H, int n_q, RowStrides sdq) {
  grid_dependency_wait();  // the main kernel's additions into dq_acc are complete
  const long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= n8) return;
  const long long r = i / d8;  // row (b * H + hh) * n_q + qi of the accumulator
  const long long bh = r / n_q;
  const long long dst =
      (bh / H) * sdq.b + (bh % H) * sdq.h + (r - bh * n_q) * sdq.n + (i - r * d8) * 8;
  const float4 a = reinterpret_cast<const float4*>(dq_acc)[2 * i];
  const float4 b = reinterpret_cast<const float4*>(dq_acc)[2 * i + 1];
  uint4 out;
  out.x = pack_bf16x2(a.x * scale, a.y * scale);
  out.y = pack_bf16x2(a.z * scale, a.w * scale);
  out.z = pack_bf16x2(b.x * scale, b.y * scale);
  out.w = pack_bf16x2(b.z * scale, b.w * scale);
  *reinterpret_cast<uint4*>(dq + dst) = out;
}

}  // namespace

BwdLayout bwd_layout(int B, int H, int n_q, int d) {
  BwdLayout l;
  const size_t bh = static_cast<size_t>(B) * H;
  l.num_qt = (n_q + BM - 1) / BM;
  l.cst_off = 0;
  l.dq_acc_off = bh * l.num_qt * CONST_TILE_BYTES;
  l.bytes = l.dq_acc_off + bh * static_cast<size_t>(n_q) * d * 4;
  return l;
}

namespace {

template <int D>
cudaError_t launch_bwd_d(const BwdProblem& pb, const CUtensorMap* maps, void* workspace,
                         const LaunchCtx& ctx) {
  static_assert(sizeof(Smem<D>) + 1024 <= 232448, "shared memory");
  const BwdLayout lay = bwd_layout(pb.B, pb.H, pb.n_q, D);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  uint8_t* cst = ws + lay.cst_off;
  float* dq_acc = reinterpret_cast<float*>(ws + lay.dq_acc_off);
  const long long bh = static_cast<long long>(pb.B) * pb.H;

  const long long rows = bh * static_cast<long long>(lay.num_qt) * BM;
  constexpr int rows_per_block = 256 / (D / 8);
  const long long pre_blocks = (rows + rows_per_block - 1) / rows_per_block;
  attn_bwd_pre_kernel<D><<<static_cast<unsigned>(pre_blocks), 256, 0, ctx.stream>>>(
      static_cast<const __nv_bfloat16*>(pb.o), static_cast<const __nv_bfloat16*>(pb.dout), pb.lse,
      cst, dq_acc, pb.H, pb.n_q, static_cast<int>(lay.num_qt), 1.f / pb.scale, rows, pb.so,
      pb.sdo);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;

  Params p;
  p.cst = cst;
  p.key_lens = pb.key_lens;
  p.H = pb.H;
  p.n_q = pb.n_q;
  p.n_k = pb.n_k;
  p.BH = static_cast<int>(bh);
  p.mask = pb.mask;
  p.win_left = pb.win_left;
  p.win_right = pb.win_right;
  p.num_qt = (pb.n_q + BM - 1) / BM;
  p.num_kt = (pb.n_k + BN - 1) / BN;
  p.num_items = p.BH * p.num_kt;
  p.scale_log2 = pb.scale * LOG2E;
  p.scale = pb.scale;
  p.limit_ns = ctx.limit_ns;
  p.status = ctx.status;
  const size_t smem = sizeof(Smem<D>) + 1024;
  const bool band = pb.mask == kMaskBand;
  err = cudaFuncSetAttribute(band ? reinterpret_cast<const void*>(attn_bwd_tc_kernel<true, D>)
                                  : reinterpret_cast<const void*>(attn_bwd_tc_kernel<false, D>),
                             cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (err != cudaSuccess) return err;
  const int grid = p.num_items < ctx.num_sms ? p.num_items : ctx.num_sms;
  // the main and the dQ kernels start while their predecessor drains
  // (programmatic dependent launch; each waits for it before reading its output)
  err = band ? launch_dependent(attn_bwd_tc_kernel<true, D>, dim3(grid), dim3(NUM_THREADS), smem,
                                ctx.stream, maps[0], maps[1], maps[2], maps[3], maps[4], maps[5],
                                maps[6], p)
             : launch_dependent(attn_bwd_tc_kernel<false, D>, dim3(grid), dim3(NUM_THREADS), smem,
                                ctx.stream, maps[0], maps[1], maps[2], maps[3], maps[4], maps[5],
                                maps[6], p);
  if (err != cudaSuccess) return err;

  const long long n8 = bh * pb.n_q * (D / 8);
  return launch_dependent(attn_bwd_dq_kernel, dim3(static_cast<unsigned>((n8 + 255) / 256)),
                          dim3(256), 0, ctx.stream, static_cast<const float*>(dq_acc),
                          static_cast<__nv_bfloat16*>(pb.dq), pb.scale, n8, D / 8, pb.H, pb.n_q,
                          pb.sdq);
}

}  // namespace

bool bwd_head_size_ok(int d) { return d == 16 || d == 32 || d == 64; }

cudaError_t launch_bwd(const BwdProblem& pb, const CUtensorMap* maps, void* workspace,
                       const LaunchCtx& ctx) {
  switch (pb.d) {
    case 16: return launch_bwd_d<16>(pb, maps, workspace, ctx);
    case 32: return launch_bwd_d<32>(pb, maps, workspace, ctx);
    case 64: return launch_bwd_d<64>(pb, maps, workspace, ctx);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace attn
