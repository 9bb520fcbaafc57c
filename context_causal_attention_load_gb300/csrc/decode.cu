// Split-K grouped-query decode attention.
//
// "Add Pallas GPU decode attention in Maxtext inference" (MaxText pull
// request 1066), Description: decode attention (one new query token per
// sequence against the KV cache) through a grouped-query kernel.  A CTA owns
// an item (batch b, KV head g, a slice of kDecodeSplit cache positions) and
// serves all G = Hq/Hkv query heads of the group from a single read of its
// K/V rows, so the cache is streamed from HBM exactly once.
//
// Streaming: small CTAs (one warp per 32 positions), several resident per
// SM.  At entry one thread issues bulk copies (cp.async.bulk) of the
// slice's K rows with the group's q, and of its V rows, on two mbarriers, so
// the score pass starts as soon as K lands while V is still in flight.
// Compute, per warp of 32 positions: LPT lanes work on one position (each
// lane holds D/LPT columns of every head's q in registers) and form G
// partial dot products reduced with log2(LPT) shuffles.  The CTA's maximum
// per head is agreed before any exponential, so the value pass needs no
// rescaling and the lane groups' partial sums merge by plain addition in
// shared memory.  An item covering a whole sequence writes the output;
// otherwise it writes (o, m, l) and a second, small kernel merges the slices
// of each (b, g).  No atomics, no fences.
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace cpattn {

namespace {

constexpr int kWarps = kDecodeSplit / 32;  // one warp per 32 positions
constexpr int kThreads = kWarps * 32;

template <int D, int GMAX>
struct DecCfg {
  // lanes per position: keep q and o at 64 registers per lane
  static constexpr int LPT0 = D * GMAX / 64;
  static constexpr int LPT = LPT0 < 8 ? 8 : (LPT0 > 32 ? 32 : LPT0);
  static constexpr int DPL = D / LPT;   // columns per lane
  static constexpr int TPI = 32 / LPT;  // positions per warp step
  static constexpr int NSTEP = 32 / TPI;
  static constexpr int NCH = DPL >= 8 ? DPL / 8 : 1;  // 16-byte chunks per lane (DPL >= 8)
  static_assert(DPL == 4 || DPL % 8 == 0, "lane column split");
};

template <int D, int GMAX>
struct DecSmem {
  using C = DecCfg<D, GMAX>;
  // K then V; after the value pass the pair is reused for the lane groups' sums
  __nv_bfloat16 k[kDecodeSplit][D];
  __nv_bfloat16 v[kDecodeSplit][D];
  __nv_bfloat16 q[GMAX][D];
  float sc[kDecodeSplit][GMAX];  // scores (log2 domain), -inf past the cache length
  float wm[kWarps][GMAX];
  float lsum[kWarps][C::TPI][GMAX];
  uint64_t bar_k, bar_v;
  static_assert(kWarps * C::TPI * GMAX * D * 4 <= 2 * kDecodeSplit * D * 2, "partial sums fit over K and V");
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
  constexpr int LPT = C::LPT, DPL = C::DPL, TPI = C::TPI, NSTEP = C::NSTEP;
  extern __shared__ __align__(128) unsigned char smem_raw[];
  auto& sm = *reinterpret_cast<DecSmem<D, GMAX>*>(smem_raw);
  const int sp = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int max_split = gridDim.x;
  const int G = a.Hq / a.Hkv;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  int len = a.lens[b];
  if (len < 0 || len > a.Smax) {
    if (sp == 0 && g == 0 && tid == 0) atomicExch(a.err, DEV_LENS_CLAMPED);
    len = len < 0 ? 0 : a.Smax;
  }
  const int nsplit = (len + kDecodeSplit - 1) / kDecodeSplit;
  __nv_bfloat16* og = static_cast<__nv_bfloat16*>(a.out) + ((size_t)b * a.Hq + (size_t)g * G) * D;
  if (len == 0) {  // empty cache: the output is defined as zero
    if (sp == 0)
      for (int x = tid; x < G * D; x += kThreads) og[x] = __float2bfloat16(0.f);
    return;
  }
  if (sp >= nsplit) return;

  const int t0 = sp * kDecodeSplit;
  const int n = min(kDecodeSplit, len - t0);
  volatile int abort_flag = 0;
  const Abort ab{&abort_flag, a.err};
  if (tid == 0) {
    mbar_init(&sm.bar_k, 1);
    mbar_init(&sm.bar_v, 1);
    fence_mbar_init();
    const size_t row0 = ((size_t)b * a.Hkv + g) * (size_t)a.Smax + t0;
    const uint32_t bytes = (uint32_t)n * D * 2, qbytes = (uint32_t)G * D * 2;
    mbar_expect_tx(&sm.bar_k, bytes + qbytes);
    bulk_load(&sm.k[0][0], static_cast<const __nv_bfloat16*>(a.kc) + row0 * D, bytes, &sm.bar_k);
    bulk_load(&sm.q[0][0], static_cast<const __nv_bfloat16*>(a.q) + ((size_t)b * a.Hq + (size_t)g * G) * D, qbytes,
              &sm.bar_k);
    mbar_expect_tx(&sm.bar_v, bytes);
    bulk_load(&sm.v[0][0], static_cast<const __nv_bfloat16*>(a.vc) + row0 * D, bytes, &sm.bar_v);
  }
  __syncthreads();  // barriers initialised before anyone waits on them

  const int sub = lane % LPT;  // column slot within the position's lanes
  const int grp = lane / LPT;  // position slot within the warp step
  const int wbase = warp * 32;
  // ---- score pass (K) -------------------------------------------------------
  float mx[GMAX];
#pragma unroll
  for (int h = 0; h < GMAX; ++h) mx[h] = -INFINITY;
  const bool okk = mbar_wait(&sm.bar_k, 0, ab);
  {
    uint64_t q2[GMAX][DPL / 2];
#pragma unroll
    for (int h = 0; h < GMAX; ++h) {
      float x[DPL];
      load_row<D, GMAX>(&sm.q[h < G ? h : 0][0], sub, x);
#pragma unroll
      for (int j = 0; j < DPL / 2; ++j)
        q2[h][j] = h < G ? f2pack(x[2 * j] * scale_log2, x[2 * j + 1] * scale_log2) : f2pack(0.f, 0.f);
    }
#pragma unroll 4
    for (int st = 0; st < NSTEP; ++st) {
      const int tt = wbase + st * TPI + grp;
      const bool valid = okk && tt < n;
      float kx[DPL];
      load_row<D, GMAX>(&sm.k[valid ? tt : 0][0], sub, kx);
      float sv[GMAX];
#pragma unroll
      for (int h = 0; h < GMAX; ++h) {
        uint64_t acc = f2pack(0.f, 0.f);
#pragma unroll
        for (int j = 0; j < DPL / 2; ++j) acc = f2fma(q2[h][j], f2pack(kx[2 * j], kx[2 * j + 1]), acc);
        float a0, a1;
        f2unpack(acc, a0, a1);
        sv[h] = a0 + a1;
      }
#pragma unroll
      for (int off = 1; off < LPT; off <<= 1)
#pragma unroll
        for (int h = 0; h < GMAX; ++h) sv[h] += __shfl_xor_sync(0xffffffffu, sv[h], off);
#pragma unroll
      for (int h = 0; h < GMAX; ++h) {
        sv[h] = valid ? sv[h] : -INFINITY;
        mx[h] = fmaxf(mx[h], sv[h]);
        if (sub == (h % LPT)) sm.sc[tt][h] = sv[h];  // one writer per (position, head)
      }
    }
  }
  // ---- the CTA agrees on one maximum per head ---------------------------------
#pragma unroll
  for (int h = 0; h < GMAX; ++h) {
#pragma unroll
    for (int off = LPT; off < 32; off <<= 1) mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], off));
  }
  if (lane == 0)
#pragma unroll
    for (int h = 0; h < GMAX; ++h) sm.wm[warp][h] = mx[h];
  __syncthreads();
  float M[GMAX];
#pragma unroll
  for (int h = 0; h < GMAX; ++h) {
    M[h] = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M[h] = fmaxf(M[h], sm.wm[w][h]);
  }
  // ---- value pass (V) -------------------------------------------------------
  uint64_t o2[GMAX][DPL / 2];
  float l[GMAX];
#pragma unroll
  for (int h = 0; h < GMAX; ++h) {
    l[h] = 0.f;
#pragma unroll
    for (int j = 0; j < DPL / 2; ++j) o2[h][j] = f2pack(0.f, 0.f);
  }
  const bool okv = mbar_wait(&sm.bar_v, 0, ab);
#pragma unroll 4
  for (int st = 0; st < NSTEP; ++st) {
    const int tt = wbase + st * TPI + grp;
    const bool valid = okv && tt < n;
    float vx[DPL];
    load_row<D, GMAX>(&sm.v[valid ? tt : 0][0], sub, vx);
#pragma unroll
    for (int h = 0; h < GMAX; ++h) {
      const float p = valid ? fast_exp2(sm.sc[tt][h] - M[h]) : 0.f;
      l[h] += p;
      const uint64_t p2 = f2pack(p, p);
#pragma unroll
      for (int j = 0; j < DPL / 2; ++j) o2[h][j] = f2fma(p2, f2pack(vx[2 * j], vx[2 * j + 1]), o2[h][j]);
    }
  }
  __syncthreads();  // K and V are dead: their space takes the partial sums
  float* part = reinterpret_cast<float*>(&sm.k[0][0]);  // [kWarps][TPI][GMAX][D]
#pragma unroll
  for (int h = 0; h < GMAX; ++h) {
    float* dst = part + ((size_t)(warp * TPI + grp) * GMAX + h) * D;
#pragma unroll
    for (int j = 0; j < DPL / 2; ++j) {
      float x0, x1;
      f2unpack(o2[h][j], x0, x1);
      dst[col_of<D, GMAX>(sub, 2 * j)] = x0;
      dst[col_of<D, GMAX>(sub, 2 * j + 1)] = x1;
    }
    if (sub == 0) sm.lsum[warp][grp][h] = l[h];
  }
  __syncthreads();
  const int bg = b * a.Hkv + g;
  for (int x = tid; x < G * D; x += kThreads) {
    const int h = x / D, d = x - h * D;
    float acc = 0.f, L = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps * TPI; ++w) {
      acc += part[((size_t)w * GMAX + h) * D + d];
      L += sm.lsum[w / TPI][w % TPI][h];
    }
    if (nsplit == 1) {
      og[x] = __float2bfloat16(acc / L);
    } else {
      a.part_o[(((size_t)bg * max_split + sp) * GMAX + h) * D + d] = acc;
      if (d == 0) {
        float* ml = a.part_ml + (((size_t)bg * max_split + sp) * GMAX + h) * 2;
        ml[0] = M[h];
        ml[1] = L;
      }
    }
  }
}

// merge the slices of every (b, g) that has more than one: one CTA per (b, g)
template <int D, int GMAX>
__global__ void __launch_bounds__(128) gqa_decode_combine_kernel(DecodeArgs a, int max_split) {
  const int bg = blockIdx.x;
  const int b = bg / a.Hkv, g = bg - b * a.Hkv;
  const int G = a.Hq / a.Hkv;
  int len = a.lens[b];
  len = len < 0 ? 0 : (len > a.Smax ? a.Smax : len);
  const int nsplit = (len + kDecodeSplit - 1) / kDecodeSplit;
  if (nsplit <= 1) return;
  __shared__ float cm[GMAX], cl[GMAX];
  const int tid = threadIdx.x;
  if (tid < G) {
    float M = -INFINITY;
    for (int s2 = 0; s2 < nsplit; ++s2) M = fmaxf(M, a.part_ml[(((size_t)bg * max_split + s2) * GMAX + tid) * 2]);
    float L = 0.f;
    for (int s2 = 0; s2 < nsplit; ++s2) {
      const float* ml = a.part_ml + (((size_t)bg * max_split + s2) * GMAX + tid) * 2;
      L += ml[1] * fast_exp2(ml[0] - M);
    }
    cm[tid] = M;
    cl[tid] = L;
  }
  __syncthreads();
  __nv_bfloat16* og = static_cast<__nv_bfloat16*>(a.out) + ((size_t)b * a.Hq + (size_t)g * G) * D;
  for (int x = tid; x < G * D; x += 128) {
    const int h = x / D, d = x - h * D;
    float acc = 0.f;
    for (int s2 = 0; s2 < nsplit; ++s2) {
      const float m2 = a.part_ml[(((size_t)bg * max_split + s2) * GMAX + h) * 2];
      acc = fmaf(a.part_o[(((size_t)bg * max_split + s2) * GMAX + h) * D + d], fast_exp2(m2 - cm[h]), acc);
    }
    og[x] = __float2bfloat16(acc / cl[h]);
  }
}

template <int D, int GMAX>
cudaError_t launch_dg(const DecodeArgs& a, cudaStream_t st) {
  const size_t smem = sizeof(DecSmem<D, GMAX>);
  auto kern = gqa_decode_kernel<D, GMAX>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const int max_split = decode_max_split(a.Smax);
  const float scale_log2 = 1.4426950408889634f / sqrtf((float)a.D);
  kern<<<dim3(max_split, a.Hkv, a.B), kThreads, smem, st>>>(a, scale_log2);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (max_split > 1) {
    gqa_decode_combine_kernel<D, GMAX><<<a.B * a.Hkv, 128, 0, st>>>(a, max_split);
    e = cudaGetLastError();
  }
  return e;
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
  return kNoAllocHeader + round256(decode_part_ml_floats(B, Hq, Hkv, Smax) * sizeof(float)) +
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
  float* ml = reinterpret_cast<float*>(p);
  p += round256(decode_part_ml_floats(B, Hq, Hkv, Smax) * sizeof(float));
  float* po = reinterpret_cast<float*>(p);
  // every slice partial the merge reads is written by the same launch
  // pair, so nothing left in the array by an earlier call is ever read
  DecodeArgs a{q, kc, vc, lens, out, B, Hq, Hkv, Smax, D, po, ml, reinterpret_cast<int*>(base)};
  return launch_gqa_decode(a, st);
}

}  // namespace cpattn
