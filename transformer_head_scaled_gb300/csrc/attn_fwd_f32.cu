// attn_fwd_f32.cu -- float32 multi-head scaled dot-product attention forward
// on the CUDA cores.
//
// Same operation as the tensor-core path (eq. (1) of "Attention Is All You
// Need", section 3.2.1, masks of section 3.2.3), for float32 tensors where
// the tensor-core path's bf16 rounding would not meet a 1e-4 tolerance.  One
// warp owns one query row and walks its visible keys 32 at a time with a
// streaming softmax in base 2 (scale*log2(e) folded into the query).  The 8
// warps of a CTA (8 query rows of one head) share the K/V tiles of 32 keys,
// staged in shared memory with asynchronous copies one tile ahead.  For the
// scores lane l takes key l of the tile (its K row and the query both read
// from shared memory with 16-byte loads); for P V, LPK = min(d, 32) lanes
// share one value row, each holding d / LPK consecutive output columns,
// 32 / LPK keys at a time.
#include "attn_internal.cuh"

namespace attn {
namespace {

constexpr int ROWS_PER_CTA = 8;  // one warp per query row
constexpr float LN2 = 0.693147180559945309f;

// 16-byte asynchronous copy global -> shared (zero-filled when !in: no byte
// is read then), so that a whole tile's copies are in flight at once.
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem, bool in) {
  const uint32_t dst = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(gmem),
               "r"(in ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

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

constexpr int KT = 32;  // keys per tile (one per lane for the scores)

// Shared memory of one CTA: K and V tiles (double-buffered), rows padded by
// 16 bytes so that the lanes' 16-byte reads of 32 different K rows spread
// over the banks; each warp's query row.
template <int D>
struct F32Smem {
  static constexpr int RS = D + 4;  // row stride in floats
  float k[2][KT][RS];
  float v[2][KT][RS];
  float q[ROWS_PER_CTA][D];
};

template <int D>
__global__ void __launch_bounds__(ROWS_PER_CTA * 32)
    attn_fwd_f32_kernel(const float* __restrict__ q, const float* __restrict__ k,
                        const float* __restrict__ v, float* __restrict__ o,
                        float* __restrict__ lse, int H, int n_q, int n_k, float scale_log2,
                        int mask, const int* __restrict__ key_lens) {
  constexpr int LPK = D < 32 ? D : 32;  // lanes per value row in P V
  constexpr int KPI = 32 / LPK;         // keys per P V step
  constexpr int DPL = D / LPK;          // output columns per lane
  extern __shared__ __align__(16) uint8_t f32_smem[];
  F32Smem<D>& sm = *reinterpret_cast<F32Smem<D>*>(f32_smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int bh = blockIdx.y;
  const int row0 = blockIdx.x * ROWS_PER_CTA;
  const int row = row0 + warp;
  const bool live = row < n_q;  // rows past n_q take part in the copies only

  int limit = n_k;
  if (mask == kMaskKeyPadding) limit = min(max(key_lens[bh / H], 0), n_k);
  int end = limit;  // keys [0, end) are visible to this row
  if (mask == kMaskCausal) end = min(end, row + 1);
  int cend = limit;  // keys this CTA needs
  if (mask == kMaskCausal) cend = min(cend, min(row0 + ROWS_PER_CTA, n_q));
  const int ntiles = (cend + KT - 1) / KT;

  const float* kb = k + static_cast<size_t>(bh) * n_k * D;
  const float* vb = v + static_cast<size_t>(bh) * n_k * D;
  // tile t into buffer t % 2: all 256 threads, 16 bytes each per copy
  auto load_tile = [&](int t) {
    const int j0 = t * KT, buf = t & 1;
#pragma unroll
    for (int e = threadIdx.x; e < KT * D / 4; e += ROWS_PER_CTA * 32) {
      const int jj = (4 * e) / D, c = (4 * e) % D;
      const bool in = j0 + jj < cend;
      const size_t off = in ? static_cast<size_t>(j0 + jj) * D + c : 0;
      cp_async16(&sm.k[buf][jj][c], kb + off, in);
      cp_async16(&sm.v[buf][jj][c], vb + off, in);
    }
    cp_async_commit();
  };
  if (ntiles > 0) load_tile(0);
  if (live) {
    const float* qp = q + (static_cast<size_t>(bh) * n_q + row) * D;
    for (int t = lane; t < D; t += 32) sm.q[warp][t] = qp[t] * scale_log2;
  }

  const int kofs = lane / LPK;        // this lane's key inside a P V step
  const int c0 = (lane % LPK) * DPL;  // and its first output column
  float m = -INFINITY, l = 0.f, acc[DPL];
#pragma unroll
  for (int c = 0; c < DPL; ++c) acc[c] = 0.f;

  for (int t = 0; t < ntiles; ++t) {
    // the next tile's copies go out before this one is awaited
    if (t + 1 < ntiles) {
      load_tile(t + 1);
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();  // tile t (and the queries) visible to every warp
    const int buf = t & 1, g0 = t * KT;
    if (live && g0 < end) {
      // ---- score of key g0 + lane (K row from shared memory, the query
      // broadcast); four independent partial sums
      const bool valid = g0 + lane < end;
      float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
#pragma unroll
      for (int c4 = 0; c4 < D / 4; ++c4) {
        const float4 kq = *reinterpret_cast<const float4*>(&sm.k[buf][lane][4 * c4]);
        const float4 qa = *reinterpret_cast<const float4*>(&sm.q[warp][4 * c4]);
        s0 = fmaf(qa.x, kq.x, s0);
        s1 = fmaf(qa.y, kq.y, s1);
        s2 = fmaf(qa.z, kq.z, s2);
        s3 = fmaf(qa.w, kq.w, s3);
      }
      const float x = valid ? (s0 + s1) + (s2 + s3) : -INFINITY;
      // ---- streaming softmax over the tile
      const float mn = fmaxf(m, warp_max(x));
      const float base = mn == -INFINITY ? 0.f : mn;
      const float alpha = exp2f(m - base);  // 0 while m = -inf
      l *= alpha;
#pragma unroll
      for (int c = 0; c < DPL; ++c) acc[c] *= alpha;
      m = mn;
      const float p = exp2f(x - base);  // 0 for keys that are not visible
      l += p;                           // per-lane partial sum, reduced at the end
      // ---- P V over the tile's visible keys
      const int nvis = min(KT, end - g0);
#pragma unroll 8
      for (int jj = 0; jj < nvis; jj += KPI) {
        const int key = jj + kofs;
        const float pj = __shfl_sync(0xffffffffu, p, key & 31);
        if (key < nvis) {
#pragma unroll
          for (int c = 0; c < DPL; ++c) acc[c] = fmaf(pj, sm.v[buf][key][c0 + c], acc[c]);
        }
      }
    }
    __syncthreads();  // every warp is done with buffer t % 2 before tile t + 2 lands there
  }
  if (!live) return;
  // lanes that took other keys of the same P V steps hold the same columns
#pragma unroll
  for (int c = 0; c < DPL; ++c)
#pragma unroll
    for (int xo = LPK; xo < 32; xo <<= 1) acc[c] += __shfl_xor_sync(0xffffffffu, acc[c], xo);
  l = warp_sum(l);
  const float inv = l > 0.f ? 1.f / l : 0.f;
  if (lane < LPK) {
    float* op = o + (static_cast<size_t>(bh) * n_q + row) * D + c0;
#pragma unroll
    for (int c = 0; c < DPL; ++c) op[c] = acc[c] * inv;
  }
  if (lane == 0 && lse != nullptr)
    lse[static_cast<size_t>(bh) * n_q + row] = l > 0.f ? (m + log2f(l)) * LN2 : -INFINITY;
}

template <int D>
cudaError_t launch_d(const Problem& pb, const LaunchCtx& ctx) {
  const size_t smem = sizeof(F32Smem<D>);
  cudaError_t err = cudaFuncSetAttribute(attn_fwd_f32_kernel<D>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
  if (err != cudaSuccess) return err;
  dim3 grid((pb.n_q + ROWS_PER_CTA - 1) / ROWS_PER_CTA, pb.B * pb.H);
  attn_fwd_f32_kernel<D><<<grid, ROWS_PER_CTA * 32, smem, ctx.stream>>>(
      static_cast<const float*>(pb.q), static_cast<const float*>(pb.k),
      static_cast<const float*>(pb.v), static_cast<float*>(pb.o), pb.lse, pb.H, pb.n_q,
      pb.n_k, pb.scale * 1.4426950408889634f, pb.mask, pb.key_lens);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_f32(const Problem& pb, const LaunchCtx& ctx) {
  switch (pb.d) {
    case 16: return launch_d<16>(pb, ctx);
    case 32: return launch_d<32>(pb, ctx);
    case 64: return launch_d<64>(pb, ctx);
    case 128: return launch_d<128>(pb, ctx);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace attn
