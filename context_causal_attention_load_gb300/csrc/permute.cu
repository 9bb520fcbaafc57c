// Load-balance reorder of the token axis and its inverse.
//
// "Add context parallelism" (MaxText pull request 1445), Description: the
// tokens are reordered so that shard s holds chunks s and 2cp-1-s; the page
// does it with a jnp.take gather and notes that it could be improved.  In
// the [B, S, row] layout every chunk of one batch is one contiguous block of
// c*row bytes, so the gather is 2cp*B block copies.  One launch streams all
// of them with 16-byte (or the widest aligned) vectors, every warp reading
// and writing consecutive addresses: a pure HBM copy, 2 bytes moved per
// byte of tensor.
#include "common.cuh"
#include "internal.h"

namespace cpattn {

template <typename V, int UNROLL>
__global__ void __launch_bounds__(256) lb_permute_kernel(const V* __restrict__ src, V* __restrict__ dst,
                                                         long long chunk_vecs, int nchunk, int cp,
                                                         long long total, int inverse) {
  const long long stride = (long long)gridDim.x * blockDim.x;
  long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  // each thread moves UNROLL vectors per iteration, spaced by the grid
  // stride so a warp's accesses stay contiguous
  for (; i < total; i += stride * UNROLL) {
    V buf[UNROLL];
    long long so[UNROLL], dofs[UNROLL];
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) {
      long long e = i + u * stride;
      so[u] = -1;
      if (e < total) {
        long long blk = e / chunk_vecs;  // (batch, memory chunk)
        long long off = e - blk * chunk_vecs;
        long long b = blk / nchunk;
        int k = int(blk - b * nchunk);
        int s = k >> 1;
        int ch = (k & 1) ? (2 * cp - 1 - s) : s;
        long long lbpos = (b * nchunk + ch) * chunk_vecs + off;  // original-order block
        // permute: dst[slot] = src[pos];  unpermute: dst[pos] = src[slot]
        so[u] = inverse ? e : lbpos;
        dofs[u] = inverse ? lbpos : e;
      }
    }
#pragma unroll
    for (int u = 0; u < UNROLL; ++u)
      if (so[u] >= 0) buf[u] = __ldcs(src + so[u]);
#pragma unroll
    for (int u = 0; u < UNROLL; ++u)
      if (so[u] >= 0) __stcs(dst + dofs[u], buf[u]);
  }
}

template <typename V>
static cudaError_t launch_v(const void* src, void* dst, long long chunk_bytes, int nchunk, int cp,
                            int B, int inverse, int num_sms, cudaStream_t st) {
  const long long chunk_vecs = chunk_bytes / (long long)sizeof(V);
  const long long total = chunk_vecs * nchunk * (long long)B;
  constexpr int kUnroll = 4;
  long long want = (total + 256LL * kUnroll - 1) / (256LL * kUnroll);
  long long cap = (long long)num_sms * 8;  // 8 resident 256-thread blocks per SM
  int grid = int(want < cap ? want : cap);
  if (grid < 1) grid = 1;
  lb_permute_kernel<V, kUnroll><<<grid, 256, 0, st>>>(static_cast<const V*>(src), static_cast<V*>(dst),
                                                      chunk_vecs, nchunk, cp, total, inverse);
  return cudaGetLastError();
}

cudaError_t launch_lb_permute(const void* src, void* dst, int B, int S, long long row_bytes, int cp,
                              int inverse, int num_sms, cudaStream_t st) {
  const int nchunk = 2 * cp;
  const long long chunk_bytes = (long long)(S / nchunk) * row_bytes;
  const uintptr_t a = reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(dst) |
                      static_cast<uintptr_t>(chunk_bytes);
  if ((a & 15) == 0) return launch_v<uint4>(src, dst, chunk_bytes, nchunk, cp, B, inverse, num_sms, st);
  if ((a & 7) == 0) return launch_v<uint2>(src, dst, chunk_bytes, nchunk, cp, B, inverse, num_sms, st);
  if ((a & 3) == 0) return launch_v<uint32_t>(src, dst, chunk_bytes, nchunk, cp, B, inverse, num_sms, st);
  if ((a & 1) == 0) return launch_v<uint16_t>(src, dst, chunk_bytes, nchunk, cp, B, inverse, num_sms, st);
  return launch_v<uint8_t>(src, dst, chunk_bytes, nchunk, cp, B, inverse, num_sms, st);
}

}  // namespace cpattn
