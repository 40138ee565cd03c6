// attn_decode.cu -- attention of a few new queries against a key/value cache
// (the autoregressive decoding step of "Attention Is All You Need", §3.1 and
// §6.1 on "Lire << Attention Is All You Need >>": the decoder produces one
// symbol at a time; beam search keeps 4 hypotheses, each a sequence of its
// own here).
//
// Same operation as the fused forward with key padding: query i of (b, h)
// sees the keys j < cache_lens[b] of its cache; O and LSE as in eq. (1).
// With n_q <= 8 the work is a matrix-vector product per head: the kernel is
// bound by HBM bandwidth (every cached key and value is read once), so it
// runs on the CUDA cores and spends its effort on keeping the loads in
// flight: a 2-deep TMA ring of 128-key tiles per CTA, three persistent CTAs
// per SM, the ring running ahead across the heads a CTA processes.
//
// When B*h alone does not fill the GPU, the cache of each head is split into
// chunks processed by different CTAs; each writes a partial result (its own
// running max m, sum l and unnormalised O, base 2) to a workspace, and a
// second kernel merges the partials of a head (the same rescaling the online
// softmax uses between tiles).  With one chunk per head the first kernel
// writes O and LSE directly and no workspace is used.
#include <cuda_bf16.h>

#include "attn_internal.cuh"
#include "ptx.cuh"

namespace attn {
namespace {

using namespace ptx;

constexpr int DK = 64;
constexpr int KT = 128;          // keys per tile
constexpr int DSTAGES = 2;       // K/V ring depth (three CTAs per SM keep 6 tiles in flight)
constexpr int NWARPS = 4;        // each warp takes 32 keys of every tile
constexpr int THREADS = NWARPS * 32;
constexpr uint32_t TILE_BYTES = KT * DK * 2;  // 16 KB
constexpr int TAIL = 32;                        // keys per box of a partial last tile
constexpr uint32_t TAIL_BYTES = TAIL * DK * 2;  // 4 KB (a multiple of the 1 KB swizzle atom)
constexpr float LN2 = 0.693147180559945309f;
// Longest-first schedule: when the caches have lengths and there are at most
// SORT_MAX (batch entry, split) pairs, the CTAs take the work units in order
// of decreasing key count, dealt out in snake order (CTA 0..G-1, then
// G-1..0, ...), instead of round-robin by index; each CTA holds at most
// SCHED_MAX units of its own.
constexpr int SORT_MAX = 1024;
constexpr int SCHED_MAX = 32;
constexpr int NBUCKET = 64;  // key-count classes of that ordering

// Queries and per-warp partials are double-buffered by the parity of a
// unit's position in the CTA's list, so that one barrier per unit suffices.
template <int NQ>
struct __align__(1024) DecSmem {
  uint8_t k[DSTAGES][TILE_BYTES];
  uint8_t v[DSTAGES][TILE_BYTES];
  union {
    struct {
      float q[2][NQ][DK];                // queries, pre-scaled by scale*log2(e)
      float red[2][NWARPS][NQ][DK + 2];  // per-warp partials, after the tiles
    } b;
    struct {
      int count[NBUCKET];  // (batch entry, split) pairs per key-count class
      int first[NBUCKET];  // sorted position of each class's first pair
    } sort;                // before the first unit
  };
  uint64_t full[DSTAGES], empty[DSTAGES];
  int sched[SCHED_MAX];  // this CTA's units, in processing order
  int nsched;
  int abort;
};

struct DecParams {
  const __nv_bfloat16* q;
  const int* cache_lens;  // may be null: every key of the cache is valid
  __nv_bfloat16* o;
  RowStrides sq, sk, sv, so;  // element strides of q, k, v, o (batch entry, head, row)
  float* lse;
  float* part;  // workspace: [B*h][splits][n_q][DK + 2] (m, l, O), or null
  int H, BH, n_q, L_max, splits, chunk;
  int win;  // restricted self-attention: a query sees keys [L - 1 - win, L); -1: all keys
  float scale_log2;
  uint64_t limit_ns;
  int* status;
};

// Keys [begin, end) of split sp of a cache filled to L: the splits cover the
// keys the queries see, [0, L), or [L - 1 - win, L) with a window.
__device__ __forceinline__ void chunk_keys(const DecParams& p, int L, int sp, int& begin,
                                           int& end) {
  const int lo = p.win >= 0 ? max(L - 1 - p.win, 0) : 0;
  begin = lo + sp * p.chunk;
  end = min(L, begin + p.chunk);
}

// Element offset of row i of head bh (= b * H + h) in a strided tensor.
__device__ __forceinline__ long long row_off(const RowStrides& s, int bh, int H, int i) {
  return (bh / H) * s.b + (bh % H) * s.h + static_cast<long long>(i) * s.n;
}

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Resident CTAs per SM: three while their shared memory fits (228 KB per SM,
// 1 KB of it reserved per CTA, 1 KB of alignment slack each), else two.
template <int NQ>
constexpr int split_ctas() { return 3 * (sizeof(DecSmem<NQ>) + 2048) <= 233472 ? 3 : 2; }

// Persistent: CTA c processes the work units c, c + gridDim.x, ... (a unit
// is one chunk of one head's cache); thread 0 keeps the TMA ring DSTAGES
// tiles ahead across unit boundaries, so the next head's first tiles are in
// flight while the current one is finished.
template <int NQ>
__global__ void __launch_bounds__(THREADS, split_ctas<NQ>())
    attn_decode_split_kernel(const __grid_constant__ CUtensorMap tmk,
                             const __grid_constant__ CUtensorMap tmv,
                             const __grid_constant__ CUtensorMap tmk_tail,
                             const __grid_constant__ CUtensorMap tmv_tail, const DecParams p) {
  extern __shared__ uint8_t smem_raw[];
  DecSmem<NQ>& sm = *reinterpret_cast<DecSmem<NQ>*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int units = p.BH * p.splits;
  // keys [begin, end) of unit u's chunk
  auto unit_keys = [&](int u, int& bh, int& begin, int& end) {
    bh = u / p.splits;
    int L = p.L_max;
    if (p.cache_lens != nullptr) L = min(max(__ldg(p.cache_lens + bh / p.H), 0), p.L_max);
    chunk_keys(p, L, u % p.splits, begin, end);
  };

  if (threadIdx.x == 0) {
    for (int i = 0; i < DSTAGES; ++i) {
      mbar_init(smem_u32(&sm.full[i]), 1);
      mbar_init(smem_u32(&sm.empty[i]), NWARPS);
    }
    sm.abort = 0;
    fence_mbar_init();
  }

  // ---- this CTA's units.  A unit is one (batch entry, split) pair of one
  // head; the pairs are the sort keys (every head of a pair has the same
  // keys), the heads of a pair stay adjacent in the order.
  const int G = gridDim.x;
  const int pairs = (p.BH / p.H) * p.splits;
  const bool sorted =
      p.cache_lens != nullptr && pairs <= SORT_MAX && (units + G - 1) / G <= SCHED_MAX;
  if (sorted) {
    const int maxk = max(1, min(p.chunk, p.L_max));
    auto bucket_of = [&](int e) {  // key-count class of pair e (0: no key)
      const int L = min(max(__ldg(p.cache_lens + e / p.splits), 0), p.L_max);
      int begin, end;
      chunk_keys(p, L, e % p.splits, begin, end);
      const int keys = end - begin;
      return keys <= 0 ? 0 : 1 + min(NBUCKET - 2, ((keys - 1) * (NBUCKET - 1)) / maxk);
    };
    for (int i = threadIdx.x; i < NBUCKET; i += THREADS) sm.sort.count[i] = 0;
    __syncthreads();
    for (int e = threadIdx.x; e < pairs; e += THREADS) atomicAdd(&sm.sort.count[bucket_of(e)], 1);
    __syncthreads();
    if (threadIdx.x == 0) {
      int acc = 0;  // classes in decreasing order of key count
      for (int k = NBUCKET - 1; k >= 0; --k) {
        sm.sort.first[k] = acc;
        acc += sm.sort.count[k];
      }
    }
    __syncthreads();
    // unit position i*G + c (i even) or i*G + G-1-c (i odd) of the sorted
    // order; inside a class the pairs keep their index order
    int n_mine = 0;
    for (int i = 0; i < SCHED_MAX; ++i) {
      const int pos = i * G + ((i & 1) ? G - 1 - static_cast<int>(blockIdx.x) : blockIdx.x);
      if (pos >= units) break;
      n_mine = i + 1;
    }
    for (int i = warp; i < n_mine; i += NWARPS) {
      const int pos = i * G + ((i & 1) ? G - 1 - static_cast<int>(blockIdx.x) : blockIdx.x);
      const int pq = pos / p.H, hh = pos % p.H;  // sorted pair position, head
      int k = 0;
#pragma unroll 1
      for (int k0 = 0; k0 < NBUCKET; k0 += 32) {
        const int kk = k0 + lane;
        const bool hit = sm.sort.count[kk] > 0 && sm.sort.first[kk] <= pq &&
                         pq < sm.sort.first[kk] + sm.sort.count[kk];
        const unsigned m = __ballot_sync(0xffffffffu, hit);
        if (m != 0u) {
          k = k0 + __ffs(m) - 1;
          break;
        }
      }
      int rank = pq - sm.sort.first[k];  // among the pairs of class k, by index
      int e_at = 0;
#pragma unroll 1
      for (int e0 = 0; e0 < pairs; e0 += 32) {
        const int e = e0 + lane;
        unsigned m = __ballot_sync(0xffffffffu, e < pairs && bucket_of(e) == k);
        const int cnt = __popc(m);
        if (rank < cnt) {
          for (int z = 0; z < rank; ++z) m &= m - 1u;
          e_at = e0 + __ffs(m) - 1;
          break;
        }
        rank -= cnt;
      }
      if (lane == 0) {
        const int b = e_at / p.splits, sp = e_at % p.splits;
        sm.sched[i] = (b * p.H + hh) * p.splits + sp;
      }
    }
    if (threadIdx.x == 0) sm.nsched = n_mine;
  }
  __syncthreads();
  const int n_units = sorted ? sm.nsched
                             : (static_cast<int>(blockIdx.x) < units
                                    ? (units - 1 - static_cast<int>(blockIdx.x)) / G + 1
                                    : 0);
  auto unit_at = [&](int i) {  // this CTA's i-th unit (units: none left)
    if (i >= n_units) return units;
    return sorted ? sm.sched[i] : static_cast<int>(blockIdx.x) + i * G;
  };
  const volatile int* abort = &sm.abort;
  const bool producer = threadIdx.x == 0;

  // ---- producer state (thread 0): the next (unit, tile) to load
  int pi = 0, pu = unit_at(0), pt = 0, pbh = 0, pbegin = 0, pend = 0;
  if (producer && pu < units) unit_keys(pu, pbh, pbegin, pend);
  uint32_t issued = 0;
  bool pok = true;
  auto produce_one = [&]() {
    while (pu < units && pbegin + pt * KT >= pend) {
      pu = unit_at(++pi);
      pt = 0;
      if (pu < units) unit_keys(pu, pbh, pbegin, pend);
    }
    if (pu >= units || !pok) return;
    const uint32_t slot = issued % DSTAGES;
    if (issued >= DSTAGES &&
        !mbar_wait(smem_u32(&sm.empty[slot]), ((issued / DSTAGES) - 1) & 1, p.limit_ns, abort)) {
      pok = false;
      return;
    }
    const int key0 = pbegin + pt * KT;
    const int rem = pend - key0;
    const uint32_t bar = smem_u32(&sm.full[slot]);
    if (rem >= KT) {
      mbar_arrive_expect_tx(bar, 2 * TILE_BYTES);
      tma_load_4d(smem_u32(sm.k[slot]), &tmk, bar, 0, key0, pbh % p.H, pbh / p.H);
      tma_load_4d(smem_u32(sm.v[slot]), &tmv, bar, 0, key0, pbh % p.H, pbh / p.H);
    } else {
      // a partial last tile: only the 32-key boxes that hold valid keys (the
      // rows after them keep stale data, which the consumers never use)
      const int nbox = (rem + TAIL - 1) / TAIL;
      mbar_arrive_expect_tx(bar, 2 * nbox * TAIL_BYTES);
      for (int i = 0; i < nbox; ++i) {
        tma_load_4d(smem_u32(sm.k[slot]) + i * TAIL_BYTES, &tmk_tail, bar, 0, key0 + i * TAIL,
                    pbh % p.H, pbh / p.H);
        tma_load_4d(smem_u32(sm.v[slot]) + i * TAIL_BYTES, &tmv_tail, bar, 0, key0 + i * TAIL,
                    pbh % p.H, pbh / p.H);
      }
    }
    ++pt;
    ++issued;
  };
  if (producer) {
    prefetch_tmap(&tmk);
    prefetch_tmap(&tmv);
    prefetch_tmap(&tmk_tail);
    prefetch_tmap(&tmv_tail);
    for (int i = 0; i < DSTAGES; ++i) produce_one();
  }

  constexpr int QPT = (NQ * DK + THREADS - 1) / THREADS;  // query values per thread
  auto load_q = [&](int u, float (&qv)[QPT]) {
    const int bh = u / p.splits;
#pragma unroll
    for (int i = 0; i < QPT; ++i) {
      const int e = threadIdx.x + i * THREADS;
      qv[i] = (u < units && e < NQ * DK)
                  ? __bfloat162float(p.q[row_off(p.sq, bh, p.H, e / DK) + e % DK])
                  : 0.f;
    }
  };
  float qv[QPT];
  // the first unit's queries into buffer 0 (the schedule above is done with
  // the shared space: the barrier after it)
  auto store_q = [&](int buf) {
#pragma unroll
    for (int i = 0; i < QPT; ++i) {
      const int e = threadIdx.x + i * THREADS;
      if (e < NQ * DK) sm.b.q[buf][e / DK][e % DK] = qv[i] * p.scale_log2;
    }
  };
  load_q(unit_at(0), qv);
  store_q(0);
  __syncthreads();

  uint32_t consumed = 0;
  bool ok = true;
  const int r = warp * 32 + lane;  // this lane's key row inside a tile
  for (int ui = 0; ui < n_units && ok; ++ui) {
    const int u = unit_at(ui);
    const int qbuf = ui & 1;  // this unit's query and partial buffers
    int bh, begin, end;
    unit_keys(u, bh, begin, end);
    const int ntiles = end > begin ? (end - begin + KT - 1) / KT : 0;
    load_q(unit_at(ui + 1), qv);  // the next unit's queries, stored after this unit's tiles

    float m[NQ], l[NQ], o0[NQ], o1[NQ];  // this warp's running state per query
#pragma unroll
    for (int qi = 0; qi < NQ; ++qi) m[qi] = -INFINITY, l[qi] = 0.f, o0[qi] = 0.f, o1[qi] = 0.f;
    for (int t = 0; t < ntiles; ++t, ++consumed) {
      const int slot = consumed % DSTAGES;
      const uint32_t ph = (consumed / DSTAGES) & 1;
      ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&sm.full[slot]), ph, p.limit_ns, abort));
      if (!ok) break;
      // ---- scores of key r for every query (K row r, 128-byte swizzle)
      // four independent partial sums per query (short dependency chains)
      const uint8_t* krow = sm.k[slot] + r * 128;
      float s[NQ], s1[NQ], s2[NQ], s3[NQ];
#pragma unroll
      for (int qi = 0; qi < NQ; ++qi) s[qi] = s1[qi] = s2[qi] = s3[qi] = 0.f;
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const uint4 w = *reinterpret_cast<const uint4*>(krow + ((c ^ (r & 7)) << 4));
        const float kf[8] = {bf16lo(w.x), bf16hi(w.x), bf16lo(w.y), bf16hi(w.y),
                             bf16lo(w.z), bf16hi(w.z), bf16lo(w.w), bf16hi(w.w)};
#pragma unroll
        for (int qi = 0; qi < NQ; ++qi) {
          const float4 qa = *reinterpret_cast<const float4*>(&sm.b.q[qbuf][qi][c * 8]);
          const float4 qb = *reinterpret_cast<const float4*>(&sm.b.q[qbuf][qi][c * 8 + 4]);
          s[qi] = fmaf(qa.x, kf[0], s[qi]);
          s1[qi] = fmaf(qa.y, kf[1], s1[qi]);
          s2[qi] = fmaf(qa.z, kf[2], s2[qi]);
          s3[qi] = fmaf(qa.w, kf[3], s3[qi]);
          s[qi] = fmaf(qb.x, kf[4], s[qi]);
          s1[qi] = fmaf(qb.y, kf[5], s1[qi]);
          s2[qi] = fmaf(qb.z, kf[6], s2[qi]);
          s3[qi] = fmaf(qb.w, kf[7], s3[qi]);
        }
      }
#pragma unroll
      for (int qi = 0; qi < NQ; ++qi) s[qi] = (s[qi] + s1[qi]) + (s2[qi] + s3[qi]);
      const bool valid = begin + t * KT + r < end;
      // ---- online softmax over this warp's 32 keys, then P V with V row j
      float pr[NQ];
#pragma unroll
      for (int qi = 0; qi < NQ; ++qi) {
        const float sv = valid ? s[qi] : -INFINITY;
        const float mt = warp_max(sv);
        const float mn = fmaxf(m[qi], mt);
        const float base = mn == -INFINITY ? 0.f : mn;
        const float alpha = ex2(m[qi] - base);  // 0 when m = -inf
        l[qi] *= alpha;
        o0[qi] *= alpha;
        o1[qi] *= alpha;
        m[qi] = mn;
        pr[qi] = ex2(sv - base);  // 0 for invalid keys
        l[qi] += pr[qi];          // per-lane partial sum, reduced at the end
      }
      // values of keys past the cache length are never used (not even times
      // 0); even and odd keys accumulate separately (shorter chains)
      const int nvalid = min(32, max(0, end - (begin + t * KT + warp * 32)));
      float e0[NQ], e1[NQ];
#pragma unroll
      for (int qi = 0; qi < NQ; ++qi) e0[qi] = e1[qi] = 0.f;
#pragma unroll 4
      for (int j = 0; j < nvalid; j += 2) {
        const int vr = warp * 32 + j;
        const uint32_t w = *reinterpret_cast<const uint32_t*>(
            sm.v[slot] + vr * 128 + ((((lane >> 2) ^ (vr & 7)) << 4) | ((lane & 3) << 2)));
        const bool has2 = j + 1 < nvalid;
        const uint32_t w2 = has2 ? *reinterpret_cast<const uint32_t*>(
                                       sm.v[slot] + (vr + 1) * 128 +
                                       ((((lane >> 2) ^ ((vr + 1) & 7)) << 4) | ((lane & 3) << 2)))
                                 : 0u;
        const float v0 = bf16lo(w), v1 = bf16hi(w), u0 = bf16lo(w2), u1 = bf16hi(w2);
#pragma unroll
        for (int qi = 0; qi < NQ; ++qi) {
          const float pj = __shfl_sync(0xffffffffu, pr[qi], j);
          const float pk = __shfl_sync(0xffffffffu, pr[qi], (j + 1) & 31);
          o0[qi] = fmaf(pj, v0, o0[qi]);
          o1[qi] = fmaf(pj, v1, o1[qi]);
          e0[qi] = fmaf(has2 ? pk : 0.f, u0, e0[qi]);
          e1[qi] = fmaf(has2 ? pk : 0.f, u1, e1[qi]);
        }
      }
#pragma unroll
      for (int qi = 0; qi < NQ; ++qi) o0[qi] += e0[qi], o1[qi] += e1[qi];
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sm.empty[slot]));
      if (producer) produce_one();  // refill the ring (possibly from the next unit)
    }
    if (!ok) break;

    // ---- merge the four warps' states: lane sums, then across warps in smem.
    // The other buffers were last read before the previous unit's barrier,
    // which every warp has passed: the next unit's queries and this unit's
    // partials go there now, and one barrier publishes both.
    store_q(qbuf ^ 1);
#pragma unroll
    for (int qi = 0; qi < NQ; ++qi) {
      const float lw = warp_sum(l[qi]);
      sm.b.red[qbuf][warp][qi][2 * lane] = o0[qi];
      sm.b.red[qbuf][warp][qi][2 * lane + 1] = o1[qi];
      if (lane == 0) {
        sm.b.red[qbuf][warp][qi][DK] = m[qi];
        sm.b.red[qbuf][warp][qi][DK + 1] = lw;
      }
    }
    __syncthreads();
    // warp qi % NWARPS writes query qi
    for (int qi = warp; qi < NQ; qi += NWARPS) {
      float mm = -INFINITY;
#pragma unroll
      for (int w = 0; w < NWARPS; ++w) mm = fmaxf(mm, sm.b.red[qbuf][w][qi][DK]);
      const float base = mm == -INFINITY ? 0.f : mm;
      float ll = 0.f, a0 = 0.f, a1 = 0.f;
#pragma unroll
      for (int w = 0; w < NWARPS; ++w) {
        const float f = ex2(sm.b.red[qbuf][w][qi][DK] - base);
        ll += f * sm.b.red[qbuf][w][qi][DK + 1];
        a0 += f * sm.b.red[qbuf][w][qi][2 * lane];
        a1 += f * sm.b.red[qbuf][w][qi][2 * lane + 1];
      }
      const size_t row = static_cast<size_t>(bh) * NQ + qi;
      if (p.splits == 1) {
        const float inv = ll > 0.f ? 1.f / ll : 0.f;
        reinterpret_cast<uint32_t*>(p.o + row_off(p.so, bh, p.H, qi))[lane] =
            pack_bf16x2(a0 * inv, a1 * inv);
        if (lane == 0 && p.lse != nullptr)
          p.lse[row] = ll > 0.f ? (mm + __log2f(ll)) * LN2 : -INFINITY;
      } else {
        float* dst =
            p.part + ((static_cast<size_t>(bh) * p.splits + (u % p.splits)) * NQ + qi) * (DK + 2);
        dst[2 * lane] = a0;
        dst[2 * lane + 1] = a1;
        if (lane == 0) {
          dst[DK] = mm;
          dst[DK + 1] = ll;
        }
      }
    }
  }
  if (!ok || !pok) {
    if (lane == 0) atomicCAS(p.status, kDevOk, kDevTimeout);
    *reinterpret_cast<volatile int*>(&sm.abort) = 1;
  }
  // Copies still in flight land before shared memory goes away: the last
  // tile issued to each slot.
  if (producer) {
    const int never = 0;
    for (uint32_t i = 0; i < DSTAGES && i < issued; ++i) {
      const uint32_t last = i + ((issued - 1 - i) / DSTAGES) * DSTAGES;
      mbar_wait(smem_u32(&sm.full[i]), (last / DSTAGES) & 1, p.limit_ns, &never);
    }
  }
}

// The same decoding step for the head sizes 16, 32 and 128, on the CUDA cores
// with plain 16-byte loads of the cache rows (no TMA ring): one CTA of four
// warps per work unit, each warp taking every fourth group of 32 keys of the
// unit's chunk with its own online softmax (float32 P), the warps merged in
// shared memory at the end as above.  For the scores lane l takes key l of
// the group; for P V, LPK lanes share one key row, each holding DPL
// consecutive output columns, and KPI = 32 / LPK keys are taken at once.
template <int D, int NQ>
__global__ void __launch_bounds__(THREADS)
    attn_decode_rows_kernel(const __nv_bfloat16* __restrict__ kc,
                            const __nv_bfloat16* __restrict__ vc, const DecParams p) {
  constexpr int LPK = D < 32 ? D : 32;  // lanes per key row in P V
  constexpr int KPI = 32 / LPK;         // keys per P V step
  constexpr int DPL = D / LPK;          // output columns per lane
  __shared__ float sq[NQ][D];           // queries, pre-scaled by scale*log2(e)
  __shared__ float red[NWARPS][NQ][D + 2];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int u = blockIdx.x;
  const int bh = u / p.splits;
  int L = p.L_max;
  if (p.cache_lens != nullptr) L = min(max(__ldg(p.cache_lens + bh / p.H), 0), p.L_max);
  int begin, end;
  chunk_keys(p, L, u % p.splits, begin, end);
  for (int e = threadIdx.x; e < NQ * D; e += THREADS)
    sq[e / D][e % D] =
        __bfloat162float(p.q[row_off(p.sq, bh, p.H, e / D) + e % D]) * p.scale_log2;
  __syncthreads();

  const __nv_bfloat16* khead = kc + row_off(p.sk, bh, p.H, 0);  // this head's cache rows
  const __nv_bfloat16* vhead = vc + row_off(p.sv, bh, p.H, 0);
  const int kofs = lane / LPK;        // this lane's key inside a P V step
  const int c0 = (lane % LPK) * DPL;  // and its first output column
  float m[NQ], l[NQ], o[NQ][DPL];
#pragma unroll
  for (int qi = 0; qi < NQ; ++qi) {
    m[qi] = -INFINITY;
    l[qi] = 0.f;
#pragma unroll
    for (int t = 0; t < DPL; ++t) o[qi][t] = 0.f;
  }
  for (int g0 = begin + warp * 32; g0 < end; g0 += NWARPS * 32) {
    // ---- scores of key g0 + lane for every query
    const int j = g0 + lane;
    const bool valid = j < end;
    float s[NQ];
#pragma unroll
    for (int qi = 0; qi < NQ; ++qi) s[qi] = 0.f;
    if (valid) {
      const uint4* krow = reinterpret_cast<const uint4*>(khead + j * p.sk.n);
#pragma unroll
      for (int c = 0; c < D / 8; ++c) {
        const uint4 w = __ldg(krow + c);
        const float kf[8] = {bf16lo(w.x), bf16hi(w.x), bf16lo(w.y), bf16hi(w.y),
                             bf16lo(w.z), bf16hi(w.z), bf16lo(w.w), bf16hi(w.w)};
#pragma unroll
        for (int qi = 0; qi < NQ; ++qi)
#pragma unroll
          for (int e = 0; e < 8; ++e) s[qi] = fmaf(sq[qi][c * 8 + e], kf[e], s[qi]);
      }
    }
    // ---- online softmax over the group
    float pr[NQ];
#pragma unroll
    for (int qi = 0; qi < NQ; ++qi) {
      const float sv = valid ? s[qi] : -INFINITY;
      const float mn = fmaxf(m[qi], warp_max(sv));
      const float base = mn == -INFINITY ? 0.f : mn;
      const float alpha = ex2(m[qi] - base);  // 0 when m = -inf
      l[qi] *= alpha;
#pragma unroll
      for (int t = 0; t < DPL; ++t) o[qi][t] *= alpha;
      m[qi] = mn;
      pr[qi] = ex2(sv - base);  // 0 for keys past the chunk
      l[qi] += pr[qi];
    }
    // ---- P V: rows past the valid keys are never read
    const int nvalid = min(32, end - g0);
    const long long vstep = KPI * p.sv.n;
    const __nv_bfloat16* vrow = vhead + (g0 + kofs) * p.sv.n + c0;  // advanced by vstep
    if (nvalid == 32) {
      // a full group: every value this lane needs is requested before the
      // first is used (one memory round trip instead of one per key)
      constexpr int STEPS = 32 / KPI;
      constexpr int W = (DPL + 1) / 2;  // 32-bit words of DPL bf16 values
      uint32_t vw[STEPS][W];
#pragma unroll
      for (int st = 0; st < STEPS; ++st) {
        const __nv_bfloat16* vr = vrow + st * vstep;
        if constexpr (DPL == 4) {
          const uint2 w2 = __ldg(reinterpret_cast<const uint2*>(vr));
          vw[st][0] = w2.x;
          vw[st][1] = w2.y;
        } else if constexpr (DPL == 2) {
          vw[st][0] = __ldg(reinterpret_cast<const unsigned int*>(vr));
        } else {
          vw[st][0] = __ldg(reinterpret_cast<const unsigned short*>(vr));
        }
      }
#pragma unroll
      for (int st = 0; st < STEPS; ++st) {
        const int key = st * KPI + kofs;
        float vf[DPL];
#pragma unroll
        for (int t = 0; t < DPL; ++t)
          vf[t] = (t & 1) ? bf16hi(vw[st][t / 2]) : bf16lo(vw[st][t / 2]);
#pragma unroll
        for (int qi = 0; qi < NQ; ++qi) {
          const float pj = __shfl_sync(0xffffffffu, pr[qi], key);
#pragma unroll
          for (int t = 0; t < DPL; ++t) o[qi][t] = fmaf(pj, vf[t], o[qi][t]);
        }
      }
      continue;
    }
    for (int jj = 0; jj < nvalid; jj += KPI, vrow += vstep) {
      const int key = jj + kofs;
      const bool kv = key < nvalid;
      float vf[DPL];
      if (kv) {
        if constexpr (DPL == 4) {
          const uint2 w = __ldg(reinterpret_cast<const uint2*>(vrow));
          vf[0] = bf16lo(w.x), vf[1] = bf16hi(w.x), vf[2] = bf16lo(w.y), vf[3] = bf16hi(w.y);
        } else {
#pragma unroll
          for (int t = 0; t < DPL; ++t) vf[t] = __bfloat162float(vrow[t]);
        }
      } else {
#pragma unroll
        for (int t = 0; t < DPL; ++t) vf[t] = 0.f;
      }
#pragma unroll
      for (int qi = 0; qi < NQ; ++qi) {
        const float pj = __shfl_sync(0xffffffffu, pr[qi], key & 31);
#pragma unroll
        for (int t = 0; t < DPL; ++t) o[qi][t] = fmaf(kv ? pj : 0.f, vf[t], o[qi][t]);
      }
    }
  }
  // lanes that took other keys of the same P V steps hold the same columns
#pragma unroll
  for (int qi = 0; qi < NQ; ++qi)
#pragma unroll
    for (int t = 0; t < DPL; ++t)
#pragma unroll
      for (int x = LPK; x < 32; x <<= 1) o[qi][t] += __shfl_xor_sync(0xffffffffu, o[qi][t], x);
  // ---- merge the four warps' states in shared memory
#pragma unroll
  for (int qi = 0; qi < NQ; ++qi) {
    const float lw = warp_sum(l[qi]);
    if (kofs == 0) {
#pragma unroll
      for (int t = 0; t < DPL; ++t) red[warp][qi][c0 + t] = o[qi][t];
    }
    if (lane == 0) {
      red[warp][qi][D] = m[qi];
      red[warp][qi][D + 1] = lw;
    }
  }
  __syncthreads();
  for (int qi = warp; qi < NQ; qi += NWARPS) {
    float mm = -INFINITY;
#pragma unroll
    for (int w = 0; w < NWARPS; ++w) mm = fmaxf(mm, red[w][qi][D]);
    const float base = mm == -INFINITY ? 0.f : mm;
    float f[NWARPS], ll = 0.f;
#pragma unroll
    for (int w = 0; w < NWARPS; ++w) {
      f[w] = ex2(red[w][qi][D] - base);
      ll += f[w] * red[w][qi][D + 1];
    }
    const size_t row = static_cast<size_t>(bh) * NQ + qi;
    float* dst = p.splits == 1
                     ? nullptr
                     : p.part + ((static_cast<size_t>(bh) * p.splits + (u % p.splits)) * NQ + qi) *
                                    (D + 2);
    const float inv = ll > 0.f ? 1.f / ll : 0.f;
    for (int t2 = lane; t2 < D / 2; t2 += 32) {  // column pairs
      float a0 = 0.f, a1 = 0.f;
#pragma unroll
      for (int w = 0; w < NWARPS; ++w) {
        a0 += f[w] * red[w][qi][2 * t2];
        a1 += f[w] * red[w][qi][2 * t2 + 1];
      }
      if (dst == nullptr) {
        reinterpret_cast<uint32_t*>(p.o + row_off(p.so, bh, p.H, qi))[t2] =
            pack_bf16x2(a0 * inv, a1 * inv);
      } else {
        dst[2 * t2] = a0;
        dst[2 * t2 + 1] = a1;
      }
    }
    if (lane == 0) {
      if (dst == nullptr) {
        if (p.lse != nullptr) p.lse[row] = ll > 0.f ? (mm + __log2f(ll)) * LN2 : -INFINITY;
      } else {
        dst[D] = mm;
        dst[D + 1] = ll;
      }
    }
  }
}

// One warp per (b, h, query): merge the chunks' partial results.
template <int D>
__global__ void __launch_bounds__(128)
    attn_decode_combine_kernel(const float* __restrict__ part, __nv_bfloat16* __restrict__ o,
                               float* __restrict__ lse, int rows, int n_q, int splits, int H,
                               RowStrides so) {
  grid_dependency_wait();  // the split kernel's partial results are complete
  const int row = blockIdx.x * 4 + (threadIdx.x >> 5);  // (bh * n_q + qi)
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const int bh = row / n_q, qi = row % n_q;
  float mm = -INFINITY;
  for (int sp = 0; sp < splits; ++sp)
    mm = fmaxf(mm, part[((static_cast<size_t>(bh) * splits + sp) * n_q + qi) * (D + 2) + D]);
  const float base = mm == -INFINITY ? 0.f : mm;
  float ll = 0.f;
  for (int sp = 0; sp < splits; ++sp) {
    const float* src = part + ((static_cast<size_t>(bh) * splits + sp) * n_q + qi) * (D + 2);
    ll += ex2(src[D] - base) * src[D + 1];
  }
  const float inv = ll > 0.f ? 1.f / ll : 0.f;
  for (int t2 = lane; t2 < D / 2; t2 += 32) {  // column pairs
    float a0 = 0.f, a1 = 0.f;
    for (int sp = 0; sp < splits; ++sp) {
      const float* src = part + ((static_cast<size_t>(bh) * splits + sp) * n_q + qi) * (D + 2);
      const float f = ex2(src[D] - base);
      a0 += f * src[2 * t2];
      a1 += f * src[2 * t2 + 1];
    }
    reinterpret_cast<uint32_t*>(o + row_off(so, bh, H, qi))[t2] = pack_bf16x2(a0 * inv, a1 * inv);
  }
  if (lane == 0 && lse != nullptr) lse[row] = ll > 0.f ? (mm + __log2f(ll)) * LN2 : -INFINITY;
}

template <int NQ>
cudaError_t launch_split(const CUtensorMap* maps, const DecParams& p, int BH, int num_sms,
                         cudaStream_t stream) {
  const size_t smem = sizeof(DecSmem<NQ>) + 1024;
  cudaError_t err = cudaFuncSetAttribute(attn_decode_split_kernel<NQ>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
  if (err != cudaSuccess) return err;
  const int units = p.splits * BH;
  const int per_sm = split_ctas<NQ>();  // resident CTAs per SM
  const int grid = units < per_sm * num_sms ? units : per_sm * num_sms;
  attn_decode_split_kernel<NQ><<<grid, THREADS, smem, stream>>>(maps[0], maps[1], maps[2], maps[3],
                                                                  p);
  return cudaGetLastError();
}

}  // namespace

template <int D, int NQ>
cudaError_t launch_rows(const DecodeProblem& pb, const DecParams& p, int units,
                        cudaStream_t stream) {
  attn_decode_rows_kernel<D, NQ><<<units, THREADS, 0, stream>>>(
      static_cast<const __nv_bfloat16*>(pb.k_cache), static_cast<const __nv_bfloat16*>(pb.v_cache),
      p);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_rows_d(const DecodeProblem& pb, const DecParams& p, int units,
                          cudaStream_t stream) {
  switch (pb.n_q) {
    case 1: return launch_rows<D, 1>(pb, p, units, stream);
    case 2: return launch_rows<D, 2>(pb, p, units, stream);
    case 3: return launch_rows<D, 3>(pb, p, units, stream);
    case 4: return launch_rows<D, 4>(pb, p, units, stream);
    case 5: return launch_rows<D, 5>(pb, p, units, stream);
    case 6: return launch_rows<D, 6>(pb, p, units, stream);
    case 7: return launch_rows<D, 7>(pb, p, units, stream);
    case 8: return launch_rows<D, 8>(pb, p, units, stream);
    default: return cudaErrorInvalidValue;
  }
}

DecodePlan decode_plan(int B, int H, int n_q, int L_max, int d, int num_sms) {
  DecodePlan plan;
  const long long bh = static_cast<long long>(B) * H;
  const int max_tiles = (L_max + KT - 1) / KT;
  // about four units per persistent CTA (three resident per SM), so that
  // unequal cache lengths even out, and at least two tiles per chunk
  const long long want = 4LL * 3 * num_sms;
  int splits = bh >= want ? 1 : static_cast<int>((want + bh - 1) / bh);
  splits = max(1, min(splits, max(1, max_tiles / 2)));
  const int tiles_per = (max_tiles + splits - 1) / splits;
  splits = (max_tiles + tiles_per - 1) / tiles_per;
  plan.splits = splits;
  plan.chunk = tiles_per * KT;
  plan.workspace_bytes =
      splits > 1 ? static_cast<size_t>(bh) * splits * n_q * (d + 2) * sizeof(float) : 0;
  return plan;
}

cudaError_t launch_decode(const DecodeProblem& pb, const CUtensorMap* maps, const DecodePlan& plan,
                          float* workspace, const LaunchCtx& ctx) {
  DecParams p;
  p.q = static_cast<const __nv_bfloat16*>(pb.q);
  p.cache_lens = pb.cache_lens;
  p.o = static_cast<__nv_bfloat16*>(pb.o);
  p.lse = pb.lse;
  p.part = workspace;
  p.H = pb.H;
  p.BH = pb.B * pb.H;
  p.n_q = pb.n_q;
  p.L_max = pb.L_max;
  p.splits = plan.splits;
  p.chunk = plan.chunk;
  p.win = pb.window;
  p.sq = pb.sq;
  p.sk = pb.sk;
  p.sv = pb.sv;
  p.so = pb.so;
  p.scale_log2 = pb.scale * 1.4426950408889634f;
  p.limit_ns = ctx.limit_ns;
  p.status = ctx.status;
  const int BH = pb.B * pb.H;
  cudaError_t err;
  if (pb.d != DK) {
    const int units = BH * plan.splits;
    switch (pb.d) {
      case 16: err = launch_rows_d<16>(pb, p, units, ctx.stream); break;
      case 32: err = launch_rows_d<32>(pb, p, units, ctx.stream); break;
      case 128: err = launch_rows_d<128>(pb, p, units, ctx.stream); break;
      default: return cudaErrorInvalidValue;
    }
  } else switch (pb.n_q) {
    case 1: err = launch_split<1>(maps, p, BH, ctx.num_sms, ctx.stream); break;
    case 2: err = launch_split<2>(maps, p, BH, ctx.num_sms, ctx.stream); break;
    case 3: err = launch_split<3>(maps, p, BH, ctx.num_sms, ctx.stream); break;
    case 4: err = launch_split<4>(maps, p, BH, ctx.num_sms, ctx.stream); break;
    case 5: err = launch_split<5>(maps, p, BH, ctx.num_sms, ctx.stream); break;
    case 6: err = launch_split<6>(maps, p, BH, ctx.num_sms, ctx.stream); break;
    case 7: err = launch_split<7>(maps, p, BH, ctx.num_sms, ctx.stream); break;
    case 8: err = launch_split<8>(maps, p, BH, ctx.num_sms, ctx.stream); break;
    default: return cudaErrorInvalidValue;
  }
  if (err != cudaSuccess || plan.splits == 1) return err;
  const int rows = BH * pb.n_q;
  const unsigned blocks = static_cast<unsigned>((rows + 3) / 4);
  // the merge starts while the split kernel drains (programmatic dependent
  // launch; it waits for the split kernel's partials before reading them)
  auto merge = [&](auto kernel) {
    return launch_dependent(kernel, dim3(blocks), dim3(128), 0, ctx.stream,
                            static_cast<const float*>(workspace), p.o, p.lse, rows, pb.n_q,
                            plan.splits, pb.H, pb.so);
  };
  switch (pb.d) {
    case 16: return merge(attn_decode_combine_kernel<16>);
    case 32: return merge(attn_decode_combine_kernel<32>);
    case 64: return merge(attn_decode_combine_kernel<64>);
    default: return merge(attn_decode_combine_kernel<128>);
  }
}

}  // namespace attn
