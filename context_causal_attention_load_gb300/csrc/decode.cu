// Split-K grouped-query decode attention.
//
// "Add Pallas GPU decode attention in Maxtext inference" (MaxText pull
// request 1066), Description: decode attention (one new query token per
// sequence against the KV cache) through a grouped-query kernel.  Work is
// cut into items (batch b, KV head g, a slice of 128 cache positions); an
// item serves all G = Hq/Hkv query heads of the group from a single read
// of its K/V rows, so the cache is streamed from HBM exactly once.
//
// Streaming: the main kernel is persistent, one CTA per SM walking items
// cta, cta + grid, ...  A producer warp keeps several items in flight with
// bulk copies (cp.async.bulk) of the item's K rows, V rows and the group's q
// into a shared-memory ring (about 197 KB per SM for D = 128), so HBM sees
// deep, continuous, register-free concurrency while two groups of four
// compute warps take alternate items.  Compute, per warp of 32 positions: LPT lanes
// work on one position (each lane holds D/LPT columns of every head's q in
// registers), form G partial dot products, reduce them with log2(LPT)
// shuffles, and update a running (max, sum, o) per lane group with a lazy
// rescale (o is rescaled only when the maximum grows by more than 8 in the
// log2 domain).  Lane groups and warps are merged in the CTA; an item that
// covers a whole sequence writes the output, otherwise it writes its
// partial (m, l, o) and a second, small kernel merges the slices of each
// (b, g).  No atomics, no fences on the streaming path.
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace cpattn {

namespace {

constexpr int kGroupWarps = 4;                     // one item per group, 32 positions per warp
constexpr int kGroups = 2;                         // groups take alternate items
constexpr int kComputeWarps = kGroups * kGroupWarps;
constexpr int kThreads = (kComputeWarps + 1) * 32; // + one producer warp
static_assert(kGroupWarps * 32 == kDecodeSplit, "32 positions per warp");

template <int D, int GMAX>
struct DecCfg {
  // lanes per position: keep q and o at 64 registers per lane
  static constexpr int LPT0 = D * GMAX / 64;
  static constexpr int LPT = LPT0 < 8 ? 8 : (LPT0 > 32 ? 32 : LPT0);
  static constexpr int DPL = D / LPT;  // columns per lane
  static constexpr int TPI = 32 / LPT; // positions per warp step
  static constexpr int NCH = DPL >= 8 ? DPL / 8 : 1;  // 16-byte chunks per lane (DPL >= 8)
  static_assert(DPL == 4 || DPL % 8 == 0, "lane column split");
  // ring depth: as many items as fit next to the merge buffers
  static constexpr int STAGE_BYTES = 2 * kDecodeSplit * D * 2 + GMAX * D * 2;
  static constexpr int MERGE_BYTES = kComputeWarps * GMAX * (D + 2) * 4 + 1024;
  static constexpr int NST0 = (225 * 1024 - MERGE_BYTES) / STAGE_BYTES;
  static constexpr int NST = NST0 > 6 ? 6 : NST0;
  static_assert(NST >= 2, "ring of at least two items");
};

template <int D, int GMAX>
struct DecSmem {
  static constexpr int kStages = DecCfg<D, GMAX>::NST;
  __nv_bfloat16 k[kStages][kDecodeSplit][D];
  __nv_bfloat16 v[kStages][kDecodeSplit][D];
  __nv_bfloat16 q[kStages][GMAX][D];
  float wo[kComputeWarps][GMAX][D];
  float wm[kComputeWarps][GMAX];
  float wl[kComputeWarps][GMAX];
  float cm[kGroups][GMAX];
  float cl[kGroups][GMAX];
  uint64_t full[kStages];
  uint64_t empty[kStages];
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

// work item i = ((b * Hkv + g) * max_split + sp): kind 0 skip, 1 empty cache
// (write zeros), 2 attend over positions [sp*128, min(len, sp*128+128))
struct Item {
  int kind, b, g, sp, len, nsplit;
};
__device__ __forceinline__ Item decode_item(const DecodeArgs& a, int i, int max_split, bool flag_errors) {
  Item it;
  const int bg = i / max_split;
  it.sp = i - bg * max_split;
  it.b = bg / a.Hkv;
  it.g = bg - it.b * a.Hkv;
  int len = a.lens[it.b];
  if (len < 0 || len > a.Smax) {
    if (flag_errors && it.sp == 0 && it.g == 0) atomicExch(a.err, DEV_LENS_CLAMPED);
    len = len < 0 ? 0 : a.Smax;
  }
  it.len = len;
  it.nsplit = (len + kDecodeSplit - 1) / kDecodeSplit;
  it.kind = len == 0 ? (it.sp == 0 ? 1 : 0) : (it.sp < it.nsplit ? 2 : 0);
  return it;
}

__device__ __forceinline__ void group_sync(int grp) { named_bar(1 + grp, kGroupWarps * 32); }

// Persistent: each CTA walks items cta, cta + grid, ...; the producer warp
// keeps up to kStages slices in flight while the compute warps consume.
template <int D, int GMAX>
__global__ void __launch_bounds__(kThreads, 1) gqa_decode_kernel(DecodeArgs a, float scale_log2, int max_split) {
  using C = DecCfg<D, GMAX>;
  constexpr int LPT = C::LPT, DPL = C::DPL, TPI = C::TPI, kStages = C::NST;
  extern __shared__ __align__(128) unsigned char smem_raw[];
  auto& sm = *reinterpret_cast<DecSmem<D, GMAX>*>(smem_raw);
  static_assert(sizeof(DecSmem<D, GMAX>) <= 232448, "shared memory budget");
  const int G = a.Hq / a.Hkv;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int total = a.B * a.Hkv * max_split;
  const int ncta = gridDim.x, cta = blockIdx.x;
  volatile int abort_flag = 0;
  const Abort ab{&abort_flag, a.err};

  if (tid == 0) {
    for (int s2 = 0; s2 < kStages; ++s2) {
      mbar_init(&sm.full[s2], 1);
      mbar_init(&sm.empty[s2], kGroupWarps * 32);
    }
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == kComputeWarps) {
    // ---------------------------------------------------------- producer
    if (lane == 0) {
      int st = 0, ph = 0;
      for (int i = cta; i < total; i += ncta) {
        const Item it = decode_item(a, i, max_split, true);
        if (it.kind != 2) continue;
        if (!mbar_wait(&sm.empty[st], ph ^ 1, ab)) break;
        const int t0 = it.sp * kDecodeSplit;
        const int n = min(kDecodeSplit, it.len - t0);
        const uint32_t bytes = (uint32_t)n * D * 2;
        const size_t row0 = ((size_t)it.b * a.Hkv + it.g) * (size_t)a.Smax + t0;
        const uint32_t qbytes = (uint32_t)G * D * 2;
        mbar_expect_tx(&sm.full[st], 2 * bytes + qbytes);
        bulk_load(&sm.k[st][0][0], static_cast<const __nv_bfloat16*>(a.kc) + row0 * D, bytes, &sm.full[st]);
        bulk_load(&sm.v[st][0][0], static_cast<const __nv_bfloat16*>(a.vc) + row0 * D, bytes, &sm.full[st]);
        bulk_load(&sm.q[st][0][0], static_cast<const __nv_bfloat16*>(a.q) + ((size_t)it.b * a.Hq + (size_t)it.g * G) * D,
                  qbytes, &sm.full[st]);
        if (++st == kStages) { st = 0; ph ^= 1; }
      }
    }
  } else {
    // ---------------------------------------------------------- compute warps
    // Group gi (warps 4gi .. 4gi+3) takes every other loaded item.  Control
    // flow is uniform inside a group (a failed wait only skips arithmetic),
    // so its named barrier always completes.
    const int gi = warp / kGroupWarps;
    const int gw = warp % kGroupWarps;     // warp within the group
    const int gt = tid - gi * kGroupWarps * 32;
    const int sub = lane % LPT;            // column slot within the position's lanes
    const int grp = lane / LPT;            // position slot within the warp step
    int nload = 0;                         // loaded items seen so far (ring index)
    for (int i = cta; i < total; i += ncta) {
      const Item it = decode_item(a, i, max_split, false);
      if (it.kind == 0) continue;
      __nv_bfloat16* og = static_cast<__nv_bfloat16*>(a.out) + ((size_t)it.b * a.Hq + (size_t)it.g * G) * D;
      if (it.kind == 1) {  // empty cache: the output is defined as zero
        if (gi == 0)
          for (int x = gt; x < G * D; x += kGroupWarps * 32) og[x] = __float2bfloat16(0.f);
        continue;
      }
      const int n_item = nload++;
      if ((n_item % kGroups) != gi) continue;
      const int st = n_item % kStages;
      const int ph = (n_item / kStages) & 1;
      const int t0 = it.sp * kDecodeSplit;
      const int n = min(kDecodeSplit, it.len - t0);
      const bool ok = mbar_wait(&sm.full[st], ph, ab);
      // q of the group (bulk-copied with the slice) as fp32 pairs, pre-scaled to log2
      uint64_t q2[GMAX][DPL / 2];
#pragma unroll
      for (int h = 0; h < GMAX; ++h) {
        float x[DPL];
        load_row<D, GMAX>(&sm.q[st][h < G ? h : 0][0], sub, x);
#pragma unroll
        for (int j = 0; j < DPL / 2; ++j)
          q2[h][j] = h < G ? f2pack(x[2 * j] * scale_log2, x[2 * j + 1] * scale_log2) : f2pack(0.f, 0.f);
      }
      uint64_t o2[GMAX][DPL / 2];
      float m[GMAX], l[GMAX];
#pragma unroll
      for (int h = 0; h < GMAX; ++h) {
        m[h] = -INFINITY;
        l[h] = 0.f;
#pragma unroll
        for (int j = 0; j < DPL / 2; ++j) o2[h][j] = f2pack(0.f, 0.f);
      }
      const int wbase = gw * 32;
      if (ok && wbase < n) {
        const int steps = (min(32, n - wbase) + TPI - 1) / TPI;
        for (int s3 = 0; s3 < steps; ++s3) {
          const int tt = wbase + s3 * TPI + grp;  // position within the slice
          const bool valid = tt < n;
          float kx[DPL];
          load_row<D, GMAX>(&sm.k[st][valid ? tt : 0][0], sub, kx);
          float s[GMAX];
#pragma unroll
          for (int h = 0; h < GMAX; ++h) {
            uint64_t acc = f2pack(0.f, 0.f);
#pragma unroll
            for (int j = 0; j < DPL / 2; ++j) acc = f2fma(q2[h][j], f2pack(kx[2 * j], kx[2 * j + 1]), acc);
            float a0, a1;
            f2unpack(acc, a0, a1);
            s[h] = a0 + a1;
          }
#pragma unroll
          for (int off = 1; off < LPT; off <<= 1)
#pragma unroll
            for (int h = 0; h < GMAX; ++h) s[h] += __shfl_xor_sync(0xffffffffu, s[h], off);
          float vx[DPL];
          load_row<D, GMAX>(&sm.v[st][valid ? tt : 0][0], sub, vx);
#pragma unroll
          for (int h = 0; h < GMAX; ++h) {
            if (h >= G || !valid) continue;
            if (s[h] > m[h] + 8.0f) {  // lazy rescale: only when the max grows by > 2^8
              const float alpha = (m[h] == -INFINITY) ? 0.f : fast_exp2(m[h] - s[h]);
              l[h] *= alpha;
              const uint64_t a2 = f2pack(alpha, alpha);
#pragma unroll
              for (int j = 0; j < DPL / 2; ++j) o2[h][j] = f2mul(o2[h][j], a2);
              m[h] = s[h];
            }
            const float p = fast_exp2(s[h] - m[h]);
            l[h] += p;
            const uint64_t p2 = f2pack(p, p);
#pragma unroll
            for (int j = 0; j < DPL / 2; ++j) o2[h][j] = f2fma(p2, f2pack(vx[2 * j], vx[2 * j + 1]), o2[h][j]);
          }
        }
      }
      mbar_arrive(&sm.empty[st]);  // this thread is done with the slice
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
          for (int j = 0; j < DPL / 2; ++j) {
            float x0, x1;
            f2unpack(o2[h][j], x0, x1);
            const float y0 = __shfl_xor_sync(0xffffffffu, x0, off);
            const float y1 = __shfl_xor_sync(0xffffffffu, x1, off);
            o2[h][j] = f2pack(x0 * a1 + y0 * a2, x1 * a1 + y1 * a2);
          }
          m[h] = mn;
        }
      }
      if (grp == 0) {
#pragma unroll
        for (int h = 0; h < GMAX; ++h) {
#pragma unroll
          for (int j = 0; j < DPL / 2; ++j) {
            float x0, x1;
            f2unpack(o2[h][j], x0, x1);
            sm.wo[warp][h][col_of<D, GMAX>(sub, 2 * j)] = x0;
            sm.wo[warp][h][col_of<D, GMAX>(sub, 2 * j + 1)] = x1;
          }
          if (sub == 0) {
            sm.wm[warp][h] = m[h];
            sm.wl[warp][h] = l[h];
          }
        }
      }
      group_sync(gi);
      // ---- merge the group's warps --------------------------------------
      const int w0 = gi * kGroupWarps;
      if (gt < GMAX) {
        const int h = gt;
        float M = -INFINITY;
        for (int w = 0; w < kGroupWarps; ++w) M = fmaxf(M, sm.wm[w0 + w][h]);
        float L = 0.f;
        for (int w = 0; w < kGroupWarps; ++w)
          if (sm.wm[w0 + w][h] != -INFINITY) L += sm.wl[w0 + w][h] * fast_exp2(sm.wm[w0 + w][h] - M);
        sm.cm[gi][h] = M;
        sm.cl[gi][h] = L;
      }
      group_sync(gi);
      const int bg = it.b * a.Hkv + it.g;
      for (int x = gt; x < G * D; x += kGroupWarps * 32) {
        const int h = x / D, d = x - h * D;
        const float M = sm.cm[gi][h];
        float acc = 0.f;
#pragma unroll
        for (int w = 0; w < kGroupWarps; ++w)
          if (sm.wm[w0 + w][h] != -INFINITY) acc = fmaf(sm.wo[w0 + w][h][d], fast_exp2(sm.wm[w0 + w][h] - M), acc);
        if (it.nsplit == 1) og[x] = __float2bfloat16(acc / sm.cl[gi][h]);
        else a.part_o[(((size_t)bg * max_split + it.sp) * GMAX + h) * D + d] = acc;
      }
      if (it.nsplit > 1 && gt < G) {
        float* ml = a.part_ml + (((size_t)bg * max_split + it.sp) * GMAX + gt) * 2;
        ml[0] = sm.cm[gi][gt];
        ml[1] = sm.cl[gi][gt];
      }
      group_sync(gi);  // the group's merge buffers are rewritten by its next item
    }
  }
  __syncthreads();
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
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int max_split = decode_max_split(a.Smax);
  const long long items = (long long)a.B * a.Hkv * max_split;
  const int grid = (int)(items < sms ? items : sms);
  const float scale_log2 = 1.4426950408889634f / sqrtf((float)a.D);
  kern<<<grid, kThreads, smem, st>>>(a, scale_log2, max_split);
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
