// Split-K grouped-query decode attention.
//
// "Add Pallas GPU decode attention in Maxtext inference" (MaxText pull
// request 1066), Description: decode attention (one new query token per
// sequence against the KV cache) through a grouped-query kernel.  Here one
// CTA owns (batch b, KV head g, a split of 128 cache positions) and serves
// all G = Hq/Hkv query heads of the group from a single read of those K/V
// rows, so the cache is streamed from HBM exactly once.
//
// Streaming: at entry one thread issues two bulk copies (cp.async.bulk) of
// the split's K rows and V rows into shared memory (up to 64 KB in flight
// per CTA, several CTAs per SM), so HBM sees deep, register-free
// concurrency.  Compute, per warp of 32 positions: LPT lanes work on one
// position (each lane holds D/LPT columns of every head's q in registers),
// form G partial dot products, reduce them with log2(LPT) shuffles, and
// update a running (max, sum, o) per lane group with a lazy rescale (o is
// rescaled only when the maximum grows by more than 8 in the log2 domain).
// Groups, warps and finally splits are merged with the usual
// max-rescaled sums; the splits of one (b, g) are merged by the last CTA to
// finish (an arrival counter per (b, g) that this CTA resets), so the whole
// decode is one launch.
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace cpattn {

namespace {

constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
static_assert(kWarps * 32 == kDecodeSplit, "32 positions per warp");

template <int D, int GMAX>
struct DecCfg {
  // lanes per position: keep q and o at 64 registers per lane
  static constexpr int LPT0 = D * GMAX / 64;
  static constexpr int LPT = LPT0 < 8 ? 8 : (LPT0 > 32 ? 32 : LPT0);
  static constexpr int DPL = D / LPT;  // columns per lane
  static constexpr int TPI = 32 / LPT; // positions per warp step
  static constexpr int NCH = DPL >= 8 ? DPL / 8 : 1;  // 16-byte chunks per lane (DPL >= 8)
  static_assert(DPL == 4 || DPL % 8 == 0, "lane column split");
};

template <int D, int GMAX>
struct DecSmem {
  __nv_bfloat16 k[kDecodeSplit][D];
  __nv_bfloat16 v[kDecodeSplit][D];
  float wm[kWarps][GMAX];
  float wl[kWarps][GMAX];
  float wo[kWarps][GMAX][D];
  float cm[GMAX];
  float cl[GMAX];
  uint64_t bar;
  int last;
};

// the lane's columns: NCH chunks of 8 (chunk sub + j*LPT), or 4 columns when DPL == 4
template <int D, int GMAX>
__device__ __forceinline__ int col_of(int sub, int j) {
  using C = DecCfg<D, GMAX>;
  if constexpr (C::DPL == 4) return sub * 4 + j;
  else return (sub + (j >> 3) * C::LPT) * 8 + (j & 7);
}

template <int D, int GMAX>
__device__ __forceinline__ void load_row(const __nv_bfloat16* row, int sub, float (&x)[DecCfg<D, GMAX>::DPL]) {
  using C = DecCfg<D, GMAX>;
  if constexpr (C::DPL == 4) {
    const uint2 u = *reinterpret_cast<const uint2*>(row + sub * 4);
    x[0] = bf16lo(u.x); x[1] = bf16hi(u.x); x[2] = bf16lo(u.y); x[3] = bf16hi(u.y);
  } else {
#pragma unroll
    for (int j = 0; j < C::NCH; ++j) {
      const uint4 u = *reinterpret_cast<const uint4*>(row + (sub + j * C::LPT) * 8);
      x[8 * j + 0] = bf16lo(u.x); x[8 * j + 1] = bf16hi(u.x);
      x[8 * j + 2] = bf16lo(u.y); x[8 * j + 3] = bf16hi(u.y);
      x[8 * j + 4] = bf16lo(u.z); x[8 * j + 5] = bf16hi(u.z);
      x[8 * j + 6] = bf16lo(u.w); x[8 * j + 7] = bf16hi(u.w);
    }
  }
}

template <int D, int GMAX>
__global__ void __launch_bounds__(kThreads) gqa_decode_kernel(DecodeArgs a, float scale_log2) {
  using C = DecCfg<D, GMAX>;
  constexpr int LPT = C::LPT, DPL = C::DPL, TPI = C::TPI;
  extern __shared__ __align__(128) unsigned char smem_raw[];
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
  const __nv_bfloat16* qg = static_cast<const __nv_bfloat16*>(a.q) + ((size_t)b * a.Hq + (size_t)g * G) * D;
  __nv_bfloat16* og = static_cast<__nv_bfloat16*>(a.out) + ((size_t)b * a.Hq + (size_t)g * G) * D;

  if (len == 0) {  // empty cache: the output is defined as zero
    if (sp == 0)
      for (int i = tid; i < G * D; i += kThreads) og[i] = __float2bfloat16(0.f);
    return;
  }
  if (sp >= nsplit) return;

  const int t0 = sp * kDecodeSplit;
  const int n = len - t0 < kDecodeSplit ? len - t0 : kDecodeSplit;
  const size_t row0 = ((size_t)b * a.Hkv + g) * (size_t)a.Smax + t0;
  volatile int abort_flag = 0;
  const Abort ab{&abort_flag, a.err};
  if (tid == 0) {
    mbar_init(&sm.bar, 1);
    fence_mbar_init();
    const uint32_t bytes = (uint32_t)n * D * 2;
    mbar_expect_tx(&sm.bar, 2 * bytes);
    bulk_load(&sm.k[0][0], static_cast<const __nv_bfloat16*>(a.kc) + row0 * D, bytes, &sm.bar);
    bulk_load(&sm.v[0][0], static_cast<const __nv_bfloat16*>(a.vc) + row0 * D, bytes, &sm.bar);
  }

  // q of the group in registers, pre-scaled into the log2 domain
  const int sub = lane % LPT;     // column slot within the position's lanes
  const int grp = lane / LPT;     // position slot within the warp step
  float qr[GMAX][DPL];
#pragma unroll
  for (int h = 0; h < GMAX; ++h)
#pragma unroll
    for (int j = 0; j < DPL; ++j)
      qr[h][j] = h < G ? __bfloat162float(qg[h * D + col_of<D, GMAX>(sub, j)]) * scale_log2 : 0.f;

  float o[GMAX][DPL];
  float m[GMAX], l[GMAX];
#pragma unroll
  for (int h = 0; h < GMAX; ++h) {
    m[h] = -INFINITY;
    l[h] = 0.f;
#pragma unroll
    for (int j = 0; j < DPL; ++j) o[h][j] = 0.f;
  }
  __syncthreads();  // barrier initialised before anyone waits on it
  const bool ok = mbar_wait(&sm.bar, 0, ab);

  const int wbase = warp * 32;
  if (ok && wbase < n) {
    const int steps = (min(32, n - wbase) + TPI - 1) / TPI;
    for (int it = 0; it < steps; ++it) {
      const int tt = wbase + it * TPI + grp;  // position within the split
      const bool valid = tt < n;
      float kx[DPL];
      load_row<D, GMAX>(&sm.k[valid ? tt : 0][0], sub, kx);
      float s[GMAX];
#pragma unroll
      for (int h = 0; h < GMAX; ++h) {
        float acc = 0.f;
#pragma unroll
        for (int j = 0; j < DPL; ++j) acc = fmaf(qr[h][j], kx[j], acc);
        s[h] = acc;
      }
#pragma unroll
      for (int off = 1; off < LPT; off <<= 1)
#pragma unroll
        for (int h = 0; h < GMAX; ++h) s[h] += __shfl_xor_sync(0xffffffffu, s[h], off);
      float vx[DPL];
      load_row<D, GMAX>(&sm.v[valid ? tt : 0][0], sub, vx);
#pragma unroll
      for (int h = 0; h < GMAX; ++h) {
        if (h >= G || !valid) continue;
        if (s[h] > m[h] + 8.0f) {  // lazy rescale: only when the max grows by > 2^8
          const float alpha = (m[h] == -INFINITY) ? 0.f : fast_exp2(m[h] - s[h]);
          l[h] *= alpha;
#pragma unroll
          for (int j = 0; j < DPL; ++j) o[h][j] *= alpha;
          m[h] = s[h];
        }
        const float p = fast_exp2(s[h] - m[h]);
        l[h] += p;
#pragma unroll
        for (int j = 0; j < DPL; ++j) o[h][j] = fmaf(p, vx[j], o[h][j]);
      }
    }
  }
  // merge the position groups of the warp (lanes sub, sub+LPT, ...)
#pragma unroll
  for (int off = LPT; off < 32; off <<= 1) {
#pragma unroll
    for (int h = 0; h < GMAX; ++h) {
      const float mo = __shfl_xor_sync(0xffffffffu, m[h], off);
      const float lo = __shfl_xor_sync(0xffffffffu, l[h], off);
      const float mn = fmaxf(m[h], mo);
      const float a1 = (m[h] == -INFINITY) ? 0.f : fast_exp2(m[h] - mn);
      const float a2 = (mo == -INFINITY) ? 0.f : fast_exp2(mo - mn);
      l[h] = l[h] * a1 + lo * a2;
#pragma unroll
      for (int j = 0; j < DPL; ++j) {
        const float ov = __shfl_xor_sync(0xffffffffu, o[h][j], off);
        o[h][j] = o[h][j] * a1 + ov * a2;
      }
      m[h] = mn;
    }
  }
  if (grp == 0) {
#pragma unroll
    for (int h = 0; h < GMAX; ++h) {
#pragma unroll
      for (int j = 0; j < DPL; ++j) sm.wo[warp][h][col_of<D, GMAX>(sub, j)] = o[h][j];
      if (sub == 0) {
        sm.wm[warp][h] = m[h];
        sm.wl[warp][h] = l[h];
      }
    }
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
      og[i] = __float2bfloat16(acc / sm.cl[h]);
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
    og[i] = __float2bfloat16(acc / sm.cl[h]);
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

// ---------------------------------------------------------------------------
// Decode without any allocation by the library.
//
// Some callers cannot let a library call cudaMalloc: code running under an
// allocator that owns all device memory (a caching allocator or a memory pool
// sized up front), real-time serving loops that must not hit the driver's
// allocation path or its implicit synchronisation, and processes that have
// reserved nearly all of HBM for the KV cache.  For them the split partials
// and arrival counters of the decode live in this fixed, statically sized
// device array instead of library-allocated scratch.  Every GPU that loads
// the library holds the array until the process exits.
// ---------------------------------------------------------------------------
constexpr size_t kNoAllocScratchBytes = size_t(8) << 20;  // 8 MiB
constexpr size_t kNoAllocHeader = 256;                    // error word

static __device__ __align__(256) unsigned char cpattn_noalloc_scratch[kNoAllocScratchBytes];

static size_t round256(size_t x) { return (x + 255) / 256 * 256; }

size_t noalloc_decode_bytes(int B, int Hq, int Hkv, int Smax, int D) {
  return kNoAllocHeader + round256((size_t)B * Hkv * sizeof(int)) +
         round256(decode_part_ml_floats(B, Hq, Hkv, Smax) * sizeof(float)) +
         round256(decode_part_o_floats(B, Hq, Hkv, Smax, D) * sizeof(float));
}
size_t noalloc_decode_limit() { return kNoAllocScratchBytes; }

// Device address of the array, looked up once per device with that device
// current (in host code the array's name is only a host-side stand-in).
constexpr int kMaxDevices = 64;
static unsigned char* g_noalloc_ptr[kMaxDevices] = {};
static std::mutex g_noalloc_mu;

cudaError_t noalloc_scratch(int dev, unsigned char** out) {
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, cpattn_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_noalloc_ptr[dev] = static_cast<unsigned char*>(p);
  }
  *out = g_noalloc_ptr[dev];
  return cudaSuccess;
}

cudaError_t launch_gqa_decode_noalloc(const void* q, const void* kc, const void* vc, const int* lens, void* out,
                                      int B, int Hq, int Hkv, int Smax, int D, cudaStream_t st) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  unsigned char* base = nullptr;
  if ((e = noalloc_scratch(dev, &base)) != cudaSuccess) return e;
  unsigned char* p = base + kNoAllocHeader;
  int* counters = reinterpret_cast<int*>(p);
  p += round256((size_t)B * Hkv * sizeof(int));
  float* ml = reinterpret_cast<float*>(p);
  p += round256(decode_part_ml_floats(B, Hq, Hkv, Smax) * sizeof(float));
  float* po = reinterpret_cast<float*>(p);
  // the array keeps whatever the previous call left: the counters must start at zero
  if ((e = cudaMemsetAsync(counters, 0, (size_t)B * Hkv * sizeof(int), st)) != cudaSuccess) return e;
  DecodeArgs a{q, kc, vc, lens, out, B, Hq, Hkv, Smax, D, po, ml, counters, reinterpret_cast<int*>(base)};
  return launch_gqa_decode(a, st);
}

}  // namespace cpattn
