// Load-balance reorder of the token axis and its inverse.
//
// "Add context parallelism" (MaxText pull request 1445), Description: the
// tokens are reordered so that shard s holds chunks s and 2cp-1-s; the page
// does it with a jnp.take gather and notes that it could be improved.  In
// the [B, S, row] layout every chunk of one batch is one contiguous block of
// c*row bytes, so the gather is 2cp*B block copies.  One launch streams all
// of them with 16-byte (or the widest aligned) vectors, every warp reading
// and writing consecutive addresses: a pure HBM copy, 2 bytes moved per
// byte of tensor, with no per-element index arithmetic.
#include "common.cuh"
#include "internal.h"

namespace cpattn {

// blockIdx.y + gridDim.y * blockIdx.z = b * nchunk + k: memory chunk k of
// batch b, which holds original chunk chunk_of(k); the CTAs along x stream
// it.  Both block bases are computed once per CTA, so the inner loop is a
// plain strided copy.
template <typename V, int UNROLL>
__global__ void __launch_bounds__(256) lb_permute_kernel(const V* __restrict__ src, V* __restrict__ dst,
                                                         long long chunk_vecs, int nchunk, int cp, long long nblk,
                                                         int inverse) {
  const long long blk = blockIdx.y + (long long)gridDim.y * blockIdx.z;
  if (blk >= nblk) return;
  const long long b = blk / nchunk;
  const int k = int(blk - b * nchunk);
  const int s = k >> 1;
  const int ch = (k & 1) ? (2 * cp - 1 - s) : s;
  const long long slot_base = blk * chunk_vecs;
  const long long pos_base = (b * nchunk + ch) * chunk_vecs;
  // permute: dst[slot] = src[pos];  unpermute: dst[pos] = src[slot]
  const V* sp = src + (inverse ? slot_base : pos_base);
  V* dp = dst + (inverse ? pos_base : slot_base);
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < chunk_vecs; i += stride * UNROLL) {
    V buf[UNROLL];
#pragma unroll
    for (int u = 0; u < UNROLL; ++u)
      if (i + u * stride < chunk_vecs) buf[u] = __ldcs(sp + i + u * stride);
#pragma unroll
    for (int u = 0; u < UNROLL; ++u)
      if (i + u * stride < chunk_vecs) __stcs(dp + i + u * stride, buf[u]);
  }
}

template <typename V>
static cudaError_t launch_v(const void* src, void* dst, long long chunk_bytes, int nchunk, int cp,
                            int B, int inverse, int num_sms, cudaStream_t st) {
  const long long chunk_vecs = chunk_bytes / (long long)sizeof(V);
  const long long nblk = (long long)nchunk * B;
  const unsigned gy = (unsigned)(nblk < 65535 ? nblk : 65535), gz = (unsigned)((nblk + gy - 1) / gy);
  constexpr int kUnroll = 4;
  long long want = (chunk_vecs + 256LL * kUnroll - 1) / (256LL * kUnroll);
  long long cap = ((long long)num_sms * 8 + nblk - 1) / nblk;  // about 8 resident 256-thread blocks per SM
  int gx = int(want < cap ? want : cap);
  if (gx < 1) gx = 1;
  lb_permute_kernel<V, kUnroll><<<dim3(gx, gy, gz), 256, 0, st>>>(static_cast<const V*>(src), static_cast<V*>(dst),
                                                                  chunk_vecs, nchunk, cp, nblk, inverse);
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
