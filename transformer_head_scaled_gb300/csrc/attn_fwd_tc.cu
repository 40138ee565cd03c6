// attn_fwd_tc.cu -- fused multi-head scaled dot-product attention forward
// for sm_103a: TMA stages Q/K/V tiles in shared memory, tcgen05 MMAs compute
// S = Q K^T and O += P V into tensor memory, and an exp2 online softmax keeps
// the n_q x n_k score matrix on chip.
//
// What is computed is eq. (1) of "Attention Is All You Need" (section 3.2.1),
// softmax(Q K^T / sqrt(d_k)) V per head, with the forbidden connections of
// section 3.2.3 set to -inf before the softmax (causal: key j > query i;
// key padding: key j >= key_lens[b]; restricted self-attention, section 4 and
// Table 1: key j outside [i - left, i + right]).  The streaming (online) softmax is an
// exact re-association of the row softmax: the pages name it only through
// FlashAttention ("32 Transformer": exact attention without materialising
// the N x N matrix).
//
// Structure (one persistent CTA per SM, 384 threads):
//   warps 0-3  softmax of Q tile 0 (rows 0-127 of a 256-row work item),
//              one thread per row = one tensor-memory lane;
//   warps 4-7  softmax of Q tile 1 (rows 128-255);
//   warp  8    TMA producer of the Q tiles (double-buffered) and the K ring (3 deep);
//   warp  9    tensor-memory owner and MMA issuer of Q tile 0;
//   warp  10   TMA producer of the V ring (4 deep);
//   warp  11   MMA issuer of Q tile 1.
// Tensor memory (512 columns x 128 lanes x 32 bit):
//   S0 [0,128)  S1 [128,256)  O0 [256,320)  O1 [320,384)  P0 [384,448)  P1 [448,512)
// The MMA issue order per KV tile j is  PV0(j-1), S0(j), PV1(j-1), S1(j):
// while softmax 0 works on S0(j) the tensor pipe computes stage 1, and the
// reverse, so the exp work of one Q tile overlaps the MMAs of the other.
// Every wait is bounded; on timeout the kernel records kDevTimeout, all roles
// drain and the CTA returns.
#include <cuda_bf16.h>

#include "attn_internal.cuh"
#include "ptx.cuh"

namespace attn {
namespace {

using namespace ptx;

constexpr int BM = 128;      // query rows per Q tile (= tensor-memory lanes)
constexpr int QT = 2;        // Q tiles per work item
constexpr int ROWS = BM * QT;
constexpr int LOAD_WARP = 8;
constexpr int MMA_WARP = 9;
constexpr int VLOAD_WARP = 10;
constexpr int MMA1_WARP = 11;
constexpr int NUM_THREADS = 384;  // 3 warpgroups: softmax 0, softmax 1, producer + MMA
// Launched at 168 registers a thread (65536 / 384, rounded down to a multiple
// of 8); the producer warpgroup hands registers to the two softmax
// warpgroups: 2 * 184 + 136 <= 3 * 168.
constexpr int LAUNCH_REGS = 168;
constexpr uint32_t SOFTMAX_REGS = 184;
constexpr uint32_t PRODUCER_REGS = 136;
static_assert(2 * SOFTMAX_REGS + PRODUCER_REGS <= 3 * LAUNCH_REGS, "register split");
constexpr uint32_t TMEM_COLS = 512;
// Keep a stale running max until the row max has grown by more than 2^8:
// P = 2^(x - m) then stays <= 256, exact in bf16's range and harmless for
// the fp32 accumulators, and O/l is unchanged because both use the same m.
constexpr float RESCALE_THRESHOLD = 8.0f;
constexpr float LN2 = 0.693147180559945309f;

// Tile shapes per head size d (16, 32, 64, 128; d_k = d_v).  A tile row of d
// bf16 values is stored in 64-column blocks of RB bytes per row, each block
// in the widest swizzle its row fits (128, 64 or 32 bytes), the layout a TMA
// copy with that swizzle writes.  d = 128 takes 64-key K/V tiles so that S,
// O and P of both Q tiles fit the 512 tensor-memory columns.
template <int D_>
struct Cfg {
  static constexpr int D = D_;
  static constexpr int BN = D_ == 128 ? 64 : 128;          // keys per K/V tile
  static constexpr uint32_t RB = (D_ < 64 ? D_ : 64) * 2;  // bytes of a row in one block
  static constexpr int NB = D_ > 64 ? D_ / 64 : 1;          // 64-column blocks per row
  // shared-memory descriptor layout code: 2 = 128-byte, 4 = 64-byte, 6 = 32-byte swizzle
  static constexpr uint32_t SWZ = RB == 128 ? 2u : (RB == 64 ? 4u : 6u);
  static constexpr int KPB = RB / 32;                       // 16-element K steps per block row
  static constexpr int QBUF = D_ == 128 ? 1 : 2;  // Q double-buffered: the next item's Q loads early
  static constexpr int KSTAGES = 3;               // K ring depth
  static constexpr int VSTAGES = D_ == 128 ? 3 : 4;  // V is held about two tiles longer than K
  static constexpr uint32_t Q_TILE = BM * D_ * 2;    // a Q (or O) tile
  static constexpr uint32_t KV_TILE = BN * D_ * 2;   // a K or V tile
  static constexpr uint32_t Q_BLOCK = BM * RB;       // one column block of a Q tile
  static constexpr uint32_t KV_BLOCK = BN * RB;
  static constexpr uint32_t OW = D_ < 32 ? 32 : D_;  // tensor-memory columns per O accumulator
  __host__ __device__ static constexpr uint32_t col_s(int s) { return BN * s; }
  __host__ __device__ static constexpr uint32_t col_o(int s) { return 2 * BN + OW * s; }
  __host__ __device__ static constexpr uint32_t col_p(int s) {
    return 2 * BN + 2 * OW + (BN / 2) * s;
  }
  // the 16-byte chunk position XOR of row r inside its swizzle atom
  __host__ __device__ static constexpr uint32_t swz(uint32_t r) {
    return ((r * RB) >> 7) & (RB / 16 - 1);
  }
  static_assert(col_p(QT) <= 512, "tensor memory");
};

template <int D_>
struct __align__(1024) Smem {
  using C = Cfg<D_>;
  uint8_t q[C::QBUF][QT][C::Q_TILE];
  uint8_t k[C::KSTAGES][C::KV_TILE];
  uint8_t v[C::VSTAGES][C::KV_TILE];
  uint8_t o[QT][C::Q_TILE];  // epilogue staging of O for the TMA store
  uint64_t q_full[C::QBUF][QT], q_empty[C::QBUF][QT];
  uint64_t k_full[C::KSTAGES], k_empty[C::KSTAGES];
  uint64_t v_full[C::VSTAGES], v_empty[C::VSTAGES];
  uint64_t s_full[QT], s_free[QT], p_full[QT], pv_done[QT];
  uint64_t drain[QT];
  uint64_t turn[QT];  // softmax ping-pong: Q tile s may run its exp phase
  uint32_t tmem_base;
  int abort;
};

struct Params {
  __nv_bfloat16* o;
  float* lse;
  const int* key_lens;
  int H, n_q, n_k, BH;
  int mask;
  int win_left, win_right;  // restricted self-attention window (band mask only)
  int num_qblocks;
  int num_items;
  float scale_log2;  // scale * log2(e): exp(scale*s) = 2^(s*scale_log2)
  uint64_t limit_ns;
  int* status;
};

// A work item: 256 query rows of one (b, h).  Its K/V tiles are j0, j0+1,
// ...; n[s] = how many of them Q tile s visits (0 when the tile lies past
// n_q or sees no key).
struct Item {
  int bh, qb;
  int key_limit;
  int j0;
  int n[QT];
};

template <bool BAND, int BN>
__device__ __forceinline__ Item decode_item(const Params& p, int t) {
  Item it;
  if (p.mask == kMaskCausal) {
    // heaviest row blocks first (longest-processing-time order)
    it.qb = p.num_qblocks - 1 - t / p.BH;
    it.bh = t % p.BH;
  } else {
    // the row blocks of one head back to back, so K/V stay hot in L2
    it.qb = t % p.num_qblocks;
    it.bh = t / p.num_qblocks;
  }
  int limit = p.n_k;
  if (p.mask == kMaskKeyPadding) {
    const int L = __ldg(p.key_lens + it.bh / p.H);
    limit = min(max(L, 0), p.n_k);
  }
  it.key_limit = limit;
  const int tiles = (limit + BN - 1) / BN;
  it.j0 = 0;
  if (BAND) {
    // the first tile of the item's stream: the lowest key of its first row's window
    it.j0 = max(it.qb * ROWS - p.win_left, 0) / BN;
  }
#pragma unroll
  for (int s = 0; s < QT; ++s) {
    const int row0 = it.qb * ROWS + s * BM;
    int n = tiles;
    if (row0 >= p.n_q) {
      n = 0;
    } else if (p.mask == kMaskCausal) {
      const int last_row = min(row0 + BM - 1, p.n_q - 1);
      n = min(tiles, last_row / BN + 1);
    } else if (BAND) {
      // tiles j0 .. the one holding the highest key of this tile's last window
      const int last_row = min(row0 + BM - 1, p.n_q - 1);
      const int lo = max(row0 - p.win_left, 0);
      const int hi = min(last_row + p.win_right, limit - 1);
      n = lo > hi ? 0 : hi / BN - it.j0 + 1;
    }
    it.n[s] = n;
  }
  return it;
}

// Shared-memory matrix descriptor (same fields as sdesc_sw128) with the
// layout code `swz` at bits 61-63.
__device__ __forceinline__ uint64_t sdesc(uint32_t smem_addr, uint32_t lbo_bytes, uint32_t sbo_bytes,
                                          uint32_t swz) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((smem_addr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>((lbo_bytes >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo_bytes >> 4) & 0x3FFFu) << 32;
  d |= 1ull << 46;
  d |= static_cast<uint64_t>(swz) << 61;
  return d;
}

template <class SmemT>
__device__ __forceinline__ void record_timeout(const Params& p, SmemT& sm) {
  atomicCAS(p.status, kDevOk, kDevTimeout);
  *reinterpret_cast<volatile int*>(&sm.abort) = 1;
}

// BAND = restricted self-attention (its own instantiation, so that the
// other masks' code is not touched by the window logic).
template <bool BAND, int D_>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    attn_fwd_tc_kernel(const __grid_constant__ CUtensorMap tmq,
                       const __grid_constant__ CUtensorMap tmk,
                       const __grid_constant__ CUtensorMap tmv,
                       const __grid_constant__ CUtensorMap tmo, const Params p) {
  using C = Cfg<D_>;
  constexpr int D = C::D, BN = C::BN, QBUF = C::QBUF, KSTAGES = C::KSTAGES,
                VSTAGES = C::VSTAGES;
  extern __shared__ uint8_t smem_raw[];
  Smem<D_>& sm = *reinterpret_cast<Smem<D_>*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const volatile int* abort = &sm.abort;

  if (threadIdx.x == 0) {
    for (int s = 0; s < QT; ++s) {
      for (int b = 0; b < QBUF; ++b) {
        mbar_init(smem_u32(&sm.q_full[b][s]), 1);
        mbar_init(smem_u32(&sm.q_empty[b][s]), 1);
      }
      mbar_init(smem_u32(&sm.s_full[s]), 1);
      mbar_init(smem_u32(&sm.s_free[s]), BM);
      mbar_init(smem_u32(&sm.p_full[s]), BM);
      mbar_init(smem_u32(&sm.pv_done[s]), 1);
    }
    for (int i = 0; i < KSTAGES; ++i) {
      mbar_init(smem_u32(&sm.k_full[i]), 1);
      mbar_init(smem_u32(&sm.k_empty[i]), QT);  // one arrival per Q tile
    }
    for (int i = 0; i < VSTAGES; ++i) {
      mbar_init(smem_u32(&sm.v_full[i]), 1);
      mbar_init(smem_u32(&sm.v_empty[i]), QT);
    }
    for (int s = 0; s < QT; ++s) mbar_init(smem_u32(&sm.drain[s]), 1);
    for (int s = 0; s < QT; ++s) mbar_init(smem_u32(&sm.turn[s]), BM);
    sm.abort = 0;
    fence_mbar_init();
  }
  if (warp == LOAD_WARP && lane == 0) {
    prefetch_tmap(&tmq);
    prefetch_tmap(&tmk);
    prefetch_tmap(&tmv);
    prefetch_tmap(&tmo);
  }
  if (warp == MMA_WARP) {
    tmem_alloc(smem_u32(&sm.tmem_base), TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;

  if (warp >= LOAD_WARP) {
    setmaxnreg_dec<PRODUCER_REGS>();
   if (warp == LOAD_WARP || warp == VLOAD_WARP) {
    // ------------------------------------------------------------ producers
    // warp 8: the Q tiles (double-buffered) and the K ring; warp 10: the V
    // ring.  Separate threads, so that a V tile waiting for a free slot never
    // holds back the K tiles (or the next Q tiles) behind it.
    if (lane == 0) {
      const bool is_v = warp == VLOAD_WARP;
      const int stages = is_v ? VSTAGES : KSTAGES;
      uint64_t* full = is_v ? sm.v_full : sm.k_full;
      uint64_t* empty = is_v ? sm.v_empty : sm.k_empty;
      uint8_t* ring = is_v ? &sm.v[0][0] : &sm.k[0][0];
      const CUtensorMap* map = is_v ? &tmv : &tmk;
      uint32_t cnt = 0;
      uint32_t items = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < p.num_items && ok; t += gridDim.x, ++items) {
        const Item it = decode_item<BAND, BN>(p, t);
        const int nmax = max(it.n[0], it.n[1]);
        // Q tiles of this item into buffer items % 2 (free once the S
        // products of item - 2 are done), then its K tiles.
        const uint32_t qb = items % QBUF, qph = (items / QBUF) & 1;
        for (int s = 0; s < QT && ok && !is_v; ++s) {
          ok = mbar_wait(smem_u32(&sm.q_empty[qb][s]), qph ^ 1, p.limit_ns, abort);
          if (!ok) break;
          const uint32_t bar = smem_u32(&sm.q_full[qb][s]);
          if (it.n[s] > 0) {
            mbar_arrive_expect_tx(bar, C::Q_TILE);
#pragma unroll
            for (int cb = 0; cb < C::NB; ++cb)
              tma_load_4d(smem_u32(sm.q[qb][s]) + cb * C::Q_BLOCK, &tmq, bar, 64 * cb,
                          it.qb * ROWS + s * BM, it.bh % p.H, it.bh / p.H);
          } else {
            mbar_arrive(bar);
          }
        }
        for (int j = 0; j < nmax && ok; ++j) {
          const uint32_t slot = cnt % stages, ph = (cnt / stages) & 1;
          ok = mbar_wait(smem_u32(&empty[slot]), ph ^ 1, p.limit_ns, abort);
          if (!ok) break;
          mbar_arrive_expect_tx(smem_u32(&full[slot]), C::KV_TILE);
#pragma unroll
          for (int cb = 0; cb < C::NB; ++cb)
            tma_load_4d(smem_u32(ring + slot * C::KV_TILE) + cb * C::KV_BLOCK, map,
                        smem_u32(&full[slot]), 64 * cb, ((BAND ? it.j0 : 0) + j) * BN,
                        it.bh % p.H, it.bh / p.H);
          ++cnt;
        }
      }
      if (!ok) {
        record_timeout(p, sm);
        // let the copies already issued land before the CTA's shared memory
        // goes away: wait (bounded, ignoring the abort flag) for the last
        // phase armed on every full barrier.
        const int never = 0;
        for (int i = 0; i < stages; ++i) {
          const uint32_t uses = cnt / stages + (static_cast<uint32_t>(i) < cnt % stages ? 1u : 0u);
          if (uses > 0) mbar_wait(smem_u32(&full[i]), (uses - 1) & 1, p.limit_ns, &never);
        }
        for (uint32_t b = 0; b < QBUF && !is_v; ++b) {
          const uint32_t uses = items / QBUF + (b < items % QBUF ? 1u : 0u);
          for (int s = 0; s < QT && uses > 0; ++s)
            mbar_wait(smem_u32(&sm.q_full[b][s]), (uses - 1) & 1, p.limit_ns, &never);
        }
      }
    }
  } else if (warp == MMA_WARP || warp == MMA1_WARP) {
    // ------------------------------------------------------------ MMA issuers
    // One issuing thread per Q tile s (warp 9: s = 0, warp 11: s = 1), so
    // that a thread blocked on a busy tensor pipe never delays the other
    // tile's products.  Tile s runs through its K/V tiles u = 0, 1, ... (all
    // items of this CTA) in the order S(0), S(1), PV(0), S(2), PV(1), ...:
    // S(u) goes as soon as the softmax has copied S(u-1) into registers
    // (s_free), PV(u-1) right after it, once P(u-1) is in tensor memory
    // (p_full).  That is the order in which these events happen, so blocking
    // waits lose nothing.  Every K/V ring slot is released by one arrival per
    // Q tile: a commit when the tile was used, a plain arrive when not.
    // The whole warp runs the control flow (so that the descriptors live in
    // uniform registers); one elected lane issues the tcgen05 operations.
    {
      const int s = warp == MMA_WARP ? 0 : 1;
      constexpr uint32_t IDESC_S = idesc_bf16_f32(BM, BN, false, false);  // Q, K both K-major
      constexpr uint32_t IDESC_O = idesc_bf16_f32(BM, D, false, true);    // V is MN-major
      constexpr uint32_t KV16 = C::KV_TILE >> 4;           // a ring slot in descriptor units
      constexpr uint32_t QBUF16 = (QT * C::Q_TILE) >> 4;   // between the Q buffers
      // K-major Q and K: 8-row groups 8*RB bytes apart; a 16-element K step
      // is 32 bytes inside a swizzled row (+2 in descriptor units), the next
      // 64-column block (d = 128) one block further.
      const uint64_t dq0 = sdesc(smem_u32(sm.q[0][s]), 16, 8 * C::RB, C::SWZ);
      const uint64_t dk = sdesc(smem_u32(sm.k[0]), 16, 8 * C::RB, C::SWZ);
      auto qstep = [](int kk) {
        return static_cast<uint32_t>((kk / C::KPB) * (C::Q_BLOCK >> 4) + (kk % C::KPB) * 2);
      };
      auto kstep = [](int kk) {
        return static_cast<uint32_t>((kk / C::KPB) * (C::KV_BLOCK >> 4) + (kk % C::KPB) * 2);
      };
      // V is the MN-major B operand: 16 keys (one K step) are 16 rows of RB
      // bytes (+RB in descriptor units); 8-row groups 8*RB bytes apart (SBO);
      // the 64-column blocks of d = 128 one block apart (LBO; with a single
      // block it is never applied).
      const uint64_t dv = sdesc(smem_u32(sm.v[0]), C::KV_BLOCK, 8 * C::RB, C::SWZ);
      const uint32_t t_s = tmem + C::col_s(s), t_o = tmem + C::col_o(s),
                     t_p = tmem + C::col_p(s);

      const bool leader = elect_one();
      bool ok = true;
      auto wait = [&](uint64_t* bar, uint32_t parity) {
        if (ok) ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(bar), parity, p.limit_ns, abort));
        return ok;
      };
      // a barrier test whose answer every lane agrees on
      auto test = [&](uint64_t* bar, uint32_t parity) {
        return __shfl_sync(0xffffffffu, mbar_test(smem_u32(bar), parity) ? 1 : 0, 0) != 0;
      };
      auto k_wait = [&](uint32_t g) { return wait(&sm.k_full[g % KSTAGES], (g / KSTAGES) & 1); };
      auto v_wait = [&](uint32_t g) { return wait(&sm.v_full[g % VSTAGES], (g / VSTAGES) & 1); };
      uint32_t u = 0;        // S products issued by this Q tile (all items)
      uint32_t npv = 0;      // PV products issued
      bool pending = false;  // the last S'd tile still owes its PV product
      uint32_t pg = 0;       // its ring index
      int pj = 0;            // its index inside its item
      // PV of the pending tile: P from tensor memory times V; an item's first
      // product overwrites O.
      auto flush_pv = [&]() {
        if (!pending || !wait(&sm.p_full[s], npv & 1) || !v_wait(pg)) return;
        tc_fence_after();
        const uint64_t b = dv + (pg % VSTAGES) * KV16;
        if (leader) {
#pragma unroll
          for (int kk = 0; kk < BN / 16; ++kk)
            mma_ts(t_o, t_p + kk * 8, b + C::RB * kk, IDESC_O, (pj > 0 || kk > 0) ? 1u : 0u);
          tc_commit(smem_u32(&sm.pv_done[s]));
          tc_commit(smem_u32(&sm.v_empty[pg % VSTAGES]));
        }
        __syncwarp();
        ++npv;
        pending = false;
      };

      uint32_t g0 = 0, items = 0;
      for (int t = blockIdx.x; t < p.num_items && ok; t += gridDim.x, ++items) {
        const Item it = decode_item<BAND, BN>(p, t);
        const int n = it.n[s];
        const int nmax = max(it.n[0], it.n[1]);
        // The previous item's last PV product goes first unless this item's
        // first S product is ready to go ahead of it.
        const uint32_t qb = items % QBUF, qph = (items / QBUF) & 1;
        const uint64_t dq = dq0 + qb * QBUF16;
        if (pending && !test(&sm.q_full[qb][s], qph)) flush_pv();
        if (!wait(&sm.q_full[qb][s], qph)) break;
        if (n == 0 && leader) tc_commit(smem_u32(&sm.q_empty[qb][s]));
        for (int j = 0; j < n && ok; ++j) {
          const uint32_t g = g0 + j;
          if (j == 0 && pending && !test(&sm.k_full[g % KSTAGES], (g / KSTAGES) & 1)) flush_pv();
          if (!k_wait(g)) break;
          if (u > 0 && !wait(&sm.s_free[s], (u - 1) & 1)) break;
          tc_fence_after();
          const uint64_t b = dk + (g % KSTAGES) * KV16;
          if (leader) {
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk)
              mma_ss(t_s, dq + qstep(kk), b + kstep(kk), IDESC_S, kk > 0 ? 1u : 0u);
            tc_commit(smem_u32(&sm.s_full[s]));
            tc_commit(smem_u32(&sm.k_empty[g % KSTAGES]));
            if (j == n - 1) tc_commit(smem_u32(&sm.q_empty[qb][s]));  // Q tile s no longer read
          }
          __syncwarp();
          ++u;
          flush_pv();  // the previous tile's PV goes right after this S product
          pending = true;
          pg = g;
          pj = j;
        }
        if (!ok) break;
        if (n < nmax) {
          // Tiles this Q tile skips: settle the pending product first (its V
          // slot may be the next one the loader needs), then release them.
          flush_pv();
          for (int j = n; j < nmax && ok; ++j) {
            const uint32_t g = g0 + j;
            if (k_wait(g) && leader) mbar_arrive(smem_u32(&sm.k_empty[g % KSTAGES]));
            if (v_wait(g) && leader) mbar_arrive(smem_u32(&sm.v_empty[g % VSTAGES]));
          }
        }
        g0 += nmax;
      }
      flush_pv();
      if (!ok && leader) record_timeout(p, sm);
      // every MMA issued by this warp completes before tensor memory is freed
      if (leader) tc_commit(smem_u32(&sm.drain[s]));
      __syncwarp();
      const int never = 0;
      mbar_wait(smem_u32(&sm.drain[s]), 0, p.limit_ns, &never);
    }
  }
  } else {
    setmaxnreg_inc<SOFTMAX_REGS>();
    // ------------------------------------------------------------ softmax
    const int s = warp >> 2;
    const int quarter = warp & 3;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t tS = tmem + lane_off + C::col_s(s);
    const uint32_t tO = tmem + lane_off + C::col_o(s);
    const uint32_t tP = tmem + lane_off + C::col_p(s);
    constexpr int SC = BN / 32;        // 32-column chunks of S
    constexpr int OC = C::OW / 32;     // 32-column chunks of O
    const bool causal = p.mask == kMaskCausal;
    constexpr bool band = BAND;
    const float c = p.scale_log2;
    uint32_t u = 0;  // tiles this stage has processed (all items)
    // Ping-pong: on the tiles both Q tiles visit, the two softmax warpgroups
    // take turns for the exp phase (the MUFU-bound part), so that one
    // group's exps overlap the other's max reduction and tensor-memory
    // traffic instead of competing for the same special-function units.
    uint32_t turns = 0;
    if (s == 1) mbar_arrive(smem_u32(&sm.turn[0]));  // Q tile 0 goes first
    bool ok = true;
    for (int t = blockIdx.x; t < p.num_items && ok; t += gridDim.x) {
      const Item it = decode_item<BAND, BN>(p, t);
      const int row0 = it.qb * ROWS + s * BM;
      const int row = row0 + quarter * 32 + lane;
      float m = -INFINITY;  // running max of scale*log2(e)*score (possibly stale)
      float l = 0.f;        // running sum of 2^(x - m)
      for (int j = 0; j < it.n[s]; ++j, ++u) {
        ok = mbar_wait(smem_u32(&sm.s_full[s]), u & 1, p.limit_ns, abort);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after();
        uint32_t r[SC][32];
#pragma unroll
        for (int q4 = 0; q4 < SC; ++q4) tmem_ld32(tS + 32 * q4, r[q4]);
        tmem_ld_wait(r[0]);
#pragma unroll
        for (int q4 = 1; q4 < SC; ++q4) reg_fence(r[q4]);
        // S is in registers: the next S product may overwrite its columns.
        tc_fence_before();
        mbar_arrive(smem_u32(&sm.s_free[s]));

        const int kbase = ((BAND ? it.j0 : 0) + j) * BN;
        if (kbase + BN > it.key_limit || (causal && kbase + BN - 1 > row0) ||
            (band && (kbase < row0 + BM - 1 - p.win_left || kbase + BN - 1 > row0 + p.win_right))) {
          int lim = it.key_limit - kbase;  // columns >= lim are forbidden
          int lo = 0;                      // and columns < lo
          if (causal) lim = min(lim, row - kbase + 1);
          if (band) {
            lim = min(lim, row + p.win_right - kbase + 1);
            lo = row - p.win_left - kbase;
          }
#pragma unroll
          for (int q4 = 0; q4 < SC; ++q4)
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (q4 * 32 + i >= lim || q4 * 32 + i < lo) r[q4][i] = __float_as_uint(-INFINITY);
        }

        float mx[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) mx[i] = -INFINITY;
#pragma unroll
        for (int q4 = 0; q4 < SC; ++q4)
#pragma unroll
          for (int i = 0; i < 32; i += 8) {
            mx[0] = max3(mx[0], __uint_as_float(r[q4][i + 0]), __uint_as_float(r[q4][i + 1]));
            mx[1] = max3(mx[1], __uint_as_float(r[q4][i + 2]), __uint_as_float(r[q4][i + 3]));
            mx[2] = max3(mx[2], __uint_as_float(r[q4][i + 4]), __uint_as_float(r[q4][i + 5]));
            mx[3] = max3(mx[3], __uint_as_float(r[q4][i + 6]), __uint_as_float(r[q4][i + 7]));
          }
        const float mt = fmaxf(max3(mx[0], mx[1], mx[2]), mx[3]) * c;

        bool rescale_o = false;
        float alpha = 1.f;
        if (mt > m + RESCALE_THRESHOLD) {
          alpha = ex2(m - mt);  // 0 when m = -inf
          l *= alpha;
          rescale_o = j > 0;
          m = mt;
        }

        const bool pingpong = j < min(it.n[0], it.n[1]);
        if (pingpong) {
          ok = __all_sync(0xffffffffu,
                          mbar_wait(smem_u32(&sm.turn[s]), turns & 1, p.limit_ns, abort));
          if (!ok) break;
        }
        const float neg_m = (m == -INFINITY) ? 0.f : -m;
        float ls0 = 0.f, ls1 = 0.f, ls2 = 0.f, ls3 = 0.f;
        uint32_t pk[SC / 2][32];
#pragma unroll
        for (int q4 = 0; q4 < SC; ++q4) {
#pragma unroll
          for (int i = 0; i < 32; i += 4) {
            float x0, x1, x2, x3;
            fma2(x0, x1, __uint_as_float(r[q4][i]), __uint_as_float(r[q4][i + 1]), c, c, neg_m,
                 neg_m);
            fma2(x2, x3, __uint_as_float(r[q4][i + 2]), __uint_as_float(r[q4][i + 3]), c, c,
                 neg_m, neg_m);
            const float p0 = ex2(x0), p1 = ex2(x1), p2 = ex2(x2), p3 = ex2(x3);
            add2(ls0, ls1, ls0, ls1, p0, p1);
            add2(ls2, ls3, ls2, ls3, p2, p3);
            pk[q4 >> 1][(q4 & 1) * 16 + (i >> 1)] = pack_bf16x2(p0, p1);
            pk[q4 >> 1][(q4 & 1) * 16 + (i >> 1) + 1] = pack_bf16x2(p2, p3);
          }
        }
        l += (ls0 + ls1) + (ls2 + ls3);
        if (pingpong) {
          mbar_arrive(smem_u32(&sm.turn[s ^ 1]));  // the other Q tile's turn
          ++turns;
        }

        // P(u) overwrites P(u-1) and O may be rescaled only once PV(u-1) is done.
        if (u > 0) {
          ok = mbar_wait(smem_u32(&sm.pv_done[s]), (u - 1) & 1, p.limit_ns, abort);
          ok = __all_sync(0xffffffffu, ok);
          if (!ok) break;
          tc_fence_after();
        }
        if (__any_sync(0xffffffffu, rescale_o)) {
          const float a = rescale_o ? alpha : 1.f;
#pragma unroll
          for (int h2 = 0; h2 < OC; ++h2) {
            uint32_t oc[32];
            tmem_ld32(tO + h2 * 32, oc);
            tmem_ld_wait(oc);
#pragma unroll
            for (int i = 0; i < 32; ++i) oc[i] = __float_as_uint(__uint_as_float(oc[i]) * a);
            tmem_st32(tO + h2 * 32, oc);
          }
        }
#pragma unroll
        for (int c2 = 0; c2 < SC / 2; ++c2) tmem_st32(tP + 32 * c2, pk[c2]);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(smem_u32(&sm.p_full[s]));
      }
      if (!ok) break;

      // ---------------------------------------------------------- epilogue
      uint32_t oreg[OC][32];
      if (it.n[s] > 0) {
        ok = mbar_wait(smem_u32(&sm.pv_done[s]), (u - 1) & 1, p.limit_ns, abort);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int h2 = 0; h2 < OC; ++h2) tmem_ld32(tO + 32 * h2, oreg[h2]);
        tmem_ld_wait(oreg[0]);
#pragma unroll
        for (int h2 = 1; h2 < OC; ++h2) reg_fence(oreg[h2]);
      } else {
#pragma unroll
        for (int h2 = 0; h2 < OC; ++h2)
#pragma unroll
          for (int i = 0; i < 32; ++i) oreg[h2][i] = 0u;
      }
      // O / l -> bf16 -> this tile's staging buffer in the swizzled layout of
      // the O tensor map -> one TMA store per 64-column block of the 128-row
      // tile (rows past n_q are clipped by the copy).
      const float inv = l > 0.f ? 1.f / l : 0.f;
      const int r_local = quarter * 32 + lane;
      const bool leader = quarter == 0 && lane == 0;
      if (leader) bulk_wait_read_all();  // the previous store has read the buffer
      named_bar_sync(1 + s, BM);
      const uint32_t rbase = smem_u32(sm.o[s]) + r_local * C::RB;
      constexpr int CPB = C::RB / 16;  // 16-byte chunks per block row
#pragma unroll
      for (int g = 0; g < D / 8; ++g) {
        const uint32_t* src = oreg[g / 4] + (g % 4) * 8;
        st_shared_v4(rbase + (g / CPB) * C::Q_BLOCK + (((g % CPB) ^ C::swz(r_local)) << 4),
                     pack_bf16x2(__uint_as_float(src[0]) * inv, __uint_as_float(src[1]) * inv),
                     pack_bf16x2(__uint_as_float(src[2]) * inv, __uint_as_float(src[3]) * inv),
                     pack_bf16x2(__uint_as_float(src[4]) * inv, __uint_as_float(src[5]) * inv),
                     pack_bf16x2(__uint_as_float(src[6]) * inv, __uint_as_float(src[7]) * inv));
      }
      fence_proxy_async_smem();
      named_bar_sync(1 + s, BM);
      if (leader && row0 < p.n_q) {
#pragma unroll
        for (int cb = 0; cb < C::NB; ++cb)
          tma_store_4d(&tmo, smem_u32(sm.o[s]) + cb * C::Q_BLOCK, 64 * cb, row0, it.bh % p.H,
                       it.bh / p.H);
        bulk_commit_group();
      }
      if (row < p.n_q && p.lse != nullptr)
        p.lse[static_cast<size_t>(it.bh) * p.n_q + row] =
            l > 0.f ? (m + __log2f(l)) * LN2 : -INFINITY;
    }
    // the last stores complete before the CTA (and its shared memory) goes away
    if (quarter == 0 && lane == 0) bulk_wait_all();
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

template <bool BAND, int D_>
cudaError_t launch_instance(const Params& p, const CUtensorMap& tmq, const CUtensorMap& tmk,
                            const CUtensorMap& tmv, const CUtensorMap& tmo, const LaunchCtx& ctx) {
  static_assert(sizeof(Smem<D_>) + 1024 <= 232448, "dynamic shared memory per CTA");
  const size_t smem = sizeof(Smem<D_>) + 1024;
  // The register hand-over inside the kernel assumes the launch holds
  // LAUNCH_REGS per thread; refuse to launch a build that does not.
  cudaFuncAttributes attr;
  cudaError_t err = cudaFuncGetAttributes(&attr, attn_fwd_tc_kernel<BAND, D_>);
  if (err != cudaSuccess) return err;
  if (attr.numRegs != LAUNCH_REGS) return cudaErrorInvalidConfiguration;
  err = cudaFuncSetAttribute(attn_fwd_tc_kernel<BAND, D_>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (err != cudaSuccess) return err;
  const int grid = p.num_items < ctx.num_sms ? p.num_items : ctx.num_sms;
  attn_fwd_tc_kernel<BAND, D_><<<grid, NUM_THREADS, smem, ctx.stream>>>(tmq, tmk, tmv, tmo, p);
  return cudaGetLastError();
}

template <int D_>
cudaError_t launch_d(const Params& p, bool band, const CUtensorMap& tmq, const CUtensorMap& tmk,
                     const CUtensorMap& tmv, const CUtensorMap& tmo, const LaunchCtx& ctx) {
  return band ? launch_instance<true, D_>(p, tmq, tmk, tmv, tmo, ctx)
              : launch_instance<false, D_>(p, tmq, tmk, tmv, tmo, ctx);
}

}  // namespace

int fwd_tc_kv_rows(int d) { return d == 128 ? Cfg<128>::BN : Cfg<64>::BN; }

cudaError_t launch_fwd_tc(const Problem& pb, const CUtensorMap& tmq, const CUtensorMap& tmk,
                          const CUtensorMap& tmv, const CUtensorMap& tmo, const LaunchCtx& ctx) {
  Params p;
  p.o = static_cast<__nv_bfloat16*>(pb.o);
  p.lse = pb.lse;
  p.key_lens = pb.key_lens;
  p.H = pb.H;
  p.n_q = pb.n_q;
  p.n_k = pb.n_k;
  p.BH = pb.B * pb.H;
  p.mask = pb.mask;
  p.win_left = pb.win_left;
  p.win_right = pb.win_right;
  p.num_qblocks = (pb.n_q + ROWS - 1) / ROWS;
  p.num_items = p.BH * p.num_qblocks;
  p.scale_log2 = pb.scale * 1.4426950408889634f;
  p.limit_ns = ctx.limit_ns;
  p.status = ctx.status;
  const bool band = pb.mask == kMaskBand;
  switch (pb.d) {
    case 16: return launch_d<16>(p, band, tmq, tmk, tmv, tmo, ctx);
    case 32: return launch_d<32>(p, band, tmq, tmk, tmv, tmo, ctx);
    case 64: return launch_d<64>(p, band, tmq, tmk, tmv, tmo, ctx);
    case 128: return launch_d<128>(p, band, tmq, tmk, tmv, tmo, ctx);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace attn
