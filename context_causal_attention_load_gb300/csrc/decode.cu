// Split-K grouped-query decode attention.
//
// "Add Pallas GPU decode attention in Maxtext inference" (MaxText pull
// request 1066), Description: decode attention (one new query token per
// sequence against the KV cache) through a grouped-query kernel.  Here one
// CTA owns (batch b, KV head g, a split of 256 cache positions) and serves
// all Hq/Hkv query heads of the group from a single read of those K/V rows,
// so the cache is streamed from HBM exactly once.  Partial results
// (running max m, sum l, unnormalised o) of the splits of one (b, g) are
// merged by the last CTA to finish (an arrival counter per (b, g), reset by
// that CTA), so the whole decode is one launch.
//
// Inside a CTA, 8 warps each take 32 positions:
//  * scores: lane = position; the lane reads its whole K row (D bf16) and
//    forms the G dot products against q held in shared memory (broadcast);
//    warp-shuffle max and sum give the warp's softmax statistics;
//  * values: lane = D/32 columns; the warp walks its 32 positions, reading
//    each V row with coalesced loads and accumulating p * v for all G heads;
//  * the 8 warps' (m, l, o) are merged in shared memory.
#include "common.cuh"
#include "internal.h"

namespace cpattn {

namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
static_assert(kWarps * 32 == kDecodeSplit, "one position per thread");

template <int D, int GMAX>
struct DecSmem {
  float q[GMAX][D];
  float p[GMAX][kDecodeSplit];
  float wm[kWarps][GMAX];
  float wl[kWarps][GMAX];
  float wo[kWarps][GMAX][D];
  float cm[GMAX];
  float cl[GMAX];
  int last;
};

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

template <int D, int GMAX>
__global__ void __launch_bounds__(kThreads) gqa_decode_kernel(DecodeArgs a, float scale_log2) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  auto& sm = *reinterpret_cast<DecSmem<D, GMAX>*>(smem_raw);
  const int sp = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int G = a.Hq / a.Hkv;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int max_split = gridDim.x;

  int len = a.lens[b];
  if (len < 0 || len > a.Smax) {
    if (sp == 0 && tid == 0) atomicExch(a.err, DEV_LENS_CLAMPED);
    len = len < 0 ? 0 : a.Smax;
  }
  const int nsplit = (len + kDecodeSplit - 1) / kDecodeSplit;
  const __nv_bfloat16* qg = static_cast<const __nv_bfloat16*>(a.q);
  __nv_bfloat16* og = static_cast<__nv_bfloat16*>(a.out);

  if (len == 0) {  // empty cache: the output is defined as zero
    if (sp == 0)
      for (int i = tid; i < G * D; i += kThreads)
        og[((size_t)b * a.Hq + (size_t)g * G) * D + i] = __float2bfloat16(0.f);
    return;
  }
  if (sp >= nsplit) return;

  // q of the group, pre-scaled into the log2 domain
  for (int i = tid; i < GMAX * D; i += kThreads) {
    int h = i / D;
    float x = 0.f;
    if (h < G) x = __bfloat162float(qg[((size_t)b * a.Hq + (size_t)g * G) * D + i]) * scale_log2;
    sm.q[h][i - h * D] = x;
  }
  __syncthreads();

  const size_t row_base = ((size_t)b * a.Hkv + g) * (size_t)a.Smax;
  const int t0 = sp * kDecodeSplit;
  const int wt0 = t0 + warp * 32;  // first position of this warp

  // ---- scores: lane = position ---------------------------------------------
  {
    const int t = wt0 + lane;
    const bool valid = t < len;
    float s[GMAX];
#pragma unroll
    for (int h = 0; h < GMAX; ++h) s[h] = 0.f;
    if (valid) {
      const uint4* kr = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(a.kc) +
                                                       (row_base + t) * D);
      constexpr int NV = D / 8;
      uint4 kv[NV];
#pragma unroll
      for (int i = 0; i < NV; ++i) kv[i] = __ldg(kr + i);
#pragma unroll
      for (int i = 0; i < NV; ++i) {
        const uint32_t w[4] = {kv[i].x, kv[i].y, kv[i].z, kv[i].w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float k0 = bf16lo(w[j]), k1 = bf16hi(w[j]);
#pragma unroll
          for (int h = 0; h < GMAX; ++h) {
            if (h < G) {
              const float2 qq = *reinterpret_cast<const float2*>(&sm.q[h][i * 8 + j * 2]);
              s[h] = fmaf(qq.x, k0, s[h]);
              s[h] = fmaf(qq.y, k1, s[h]);
            }
          }
        }
      }
    }
#pragma unroll
    for (int h = 0; h < GMAX; ++h) {
      if (h < G) {
        float sv = valid ? s[h] : -INFINITY;
        float m = warp_max(sv);
        float mref = (m == -INFINITY) ? 0.f : m;
        float p = valid ? fast_exp2(sv - mref) : 0.f;
        float l = warp_sum(p);
        sm.p[h][warp * 32 + lane] = p;
        if (lane == 0) {
          sm.wm[warp][h] = m;
          sm.wl[warp][h] = l;
        }
      }
    }
  }
  __syncwarp();

  // ---- values: lane = D/32 columns ---------------------------------------------
  {
    constexpr int C = D / 32;  // columns per lane: 4 (D=128) or 2 (D=64)
    float o[GMAX][C];
#pragma unroll
    for (int h = 0; h < GMAX; ++h)
#pragma unroll
      for (int c = 0; c < C; ++c) o[h][c] = 0.f;
    int n = len - wt0;
    n = n > 32 ? 32 : n;
    const __nv_bfloat16* vb = static_cast<const __nv_bfloat16*>(a.vc) + (row_base + wt0) * D + lane * C;
    for (int i0 = 0; i0 < n; i0 += 8) {
      uint32_t raw[8][C / 2];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        if (i0 + u < n) {
          if constexpr (C == 4) {
            uint2 x = __ldg(reinterpret_cast<const uint2*>(vb + (size_t)(i0 + u) * D));
            raw[u][0] = x.x;
            raw[u][1] = x.y;
          } else {
            raw[u][0] = __ldg(reinterpret_cast<const unsigned int*>(vb + (size_t)(i0 + u) * D));
          }
        } else {
#pragma unroll
          for (int c = 0; c < C / 2; ++c) raw[u][c] = 0u;
        }
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        float vv[C];
#pragma unroll
        for (int c = 0; c < C / 2; ++c) {
          vv[2 * c] = bf16lo(raw[u][c]);
          vv[2 * c + 1] = bf16hi(raw[u][c]);
        }
        const int pi = warp * 32 + i0 + u;
#pragma unroll
        for (int h = 0; h < GMAX; ++h) {
          if (h < G) {
            const float p = (i0 + u < n) ? sm.p[h][pi] : 0.f;
#pragma unroll
            for (int c = 0; c < C; ++c) o[h][c] = fmaf(p, vv[c], o[h][c]);
          }
        }
      }
    }
#pragma unroll
    for (int h = 0; h < GMAX; ++h)
#pragma unroll
      for (int c = 0; c < C; ++c) sm.wo[warp][h][lane * C + c] = o[h][c];
  }
  __syncthreads();

  // ---- merge the warps ---------------------------------------------------
  if (tid < GMAX) {
    const int h = tid;
    float M = -INFINITY;
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, sm.wm[w][h]);
    float L = 0.f;
    for (int w = 0; w < kWarps; ++w)
      if (sm.wm[w][h] != -INFINITY) L += sm.wl[w][h] * fast_exp2(sm.wm[w][h] - M);
    sm.cm[tid] = M;
    sm.cl[tid] = L;
  }
  __syncthreads();
  const int bg = b * a.Hkv + g;
  for (int i = tid; i < G * D; i += kThreads) {
    const int h = i / D, d = i - h * D;
    const float M = sm.cm[h];
    float acc = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w)
      if (sm.wm[w][h] != -INFINITY) acc = fmaf(sm.wo[w][h][d], fast_exp2(sm.wm[w][h] - M), acc);
    if (nsplit == 1) {
      og[((size_t)b * a.Hq + (size_t)g * G + h) * D + d] = __float2bfloat16(acc / sm.cl[h]);
    } else {
      a.part_o[(((size_t)bg * max_split + sp) * GMAX + h) * D + d] = acc;
    }
  }
  if (nsplit == 1) return;
  if (tid < G) {
    float* ml = a.part_ml + (((size_t)bg * max_split + sp) * GMAX + tid) * 2;
    ml[0] = sm.cm[tid];
    ml[1] = sm.cl[tid];
  }
  // ---- last CTA of (b, g) merges the splits ------------------------------
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    int old = atomicAdd(a.counters + bg, 1);
    sm.last = (old == nsplit - 1);
  }
  __syncthreads();
  if (!sm.last) return;
  __threadfence();
  if (tid < G) {
    float M = -INFINITY;
    for (int s2 = 0; s2 < nsplit; ++s2)
      M = fmaxf(M, __ldcg(a.part_ml + (((size_t)bg * max_split + s2) * GMAX + tid) * 2));
    float L = 0.f;
    for (int s2 = 0; s2 < nsplit; ++s2) {
      const float* ml = a.part_ml + (((size_t)bg * max_split + s2) * GMAX + tid) * 2;
      L += __ldcg(ml + 1) * fast_exp2(__ldcg(ml) - M);
    }
    sm.cm[tid] = M;
    sm.cl[tid] = L;
  }
  __syncthreads();
  for (int i = tid; i < G * D; i += kThreads) {
    const int h = i / D, d = i - h * D;
    const float M = sm.cm[h];
    float acc = 0.f;
    for (int s2 = 0; s2 < nsplit; ++s2) {
      const float m2 = __ldcg(a.part_ml + (((size_t)bg * max_split + s2) * GMAX + h) * 2);
      acc = fmaf(__ldcg(a.part_o + (((size_t)bg * max_split + s2) * GMAX + h) * D + d), fast_exp2(m2 - M), acc);
    }
    og[((size_t)b * a.Hq + (size_t)g * G + h) * D + d] = __float2bfloat16(acc / sm.cl[h]);
  }
  if (tid == 0) a.counters[bg] = 0;  // ready for the next launch
}

template <int D, int GMAX>
cudaError_t launch_dg(const DecodeArgs& a, cudaStream_t st) {
  const size_t smem = sizeof(DecSmem<D, GMAX>);
  auto kern = gqa_decode_kernel<D, GMAX>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid(decode_max_split(a.Smax), a.Hkv, a.B);
  const float scale_log2 = 1.4426950408889634f / sqrtf((float)a.D);
  kern<<<grid, kThreads, smem, st>>>(a, scale_log2);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_d(const DecodeArgs& a, cudaStream_t st) {
  const int G = a.Hq / a.Hkv;
  if (G <= 1) return launch_dg<D, 1>(a, st);
  if (G <= 2) return launch_dg<D, 2>(a, st);
  if (G <= 4) return launch_dg<D, 4>(a, st);
  if (G <= 8) return launch_dg<D, 8>(a, st);
  return launch_dg<D, 16>(a, st);
}

}  // namespace

int decode_max_split(int Smax) { return (Smax + kDecodeSplit - 1) / kDecodeSplit; }

static int gmax_of(int G) { return G <= 1 ? 1 : G <= 2 ? 2 : G <= 4 ? 4 : G <= 8 ? 8 : 16; }

size_t decode_part_o_floats(int B, int Hq, int Hkv, int Smax, int D) {
  return (size_t)B * Hkv * decode_max_split(Smax) * gmax_of(Hq / Hkv) * D;
}
size_t decode_part_ml_floats(int B, int Hq, int Hkv, int Smax) {
  return (size_t)B * Hkv * decode_max_split(Smax) * gmax_of(Hq / Hkv) * 2;
}

cudaError_t launch_gqa_decode(const DecodeArgs& a, cudaStream_t st) {
  if (a.D == 128) return launch_d<128>(a, st);
  return launch_d<64>(a, st);
}

}  // namespace cpattn
