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

#include <cuda_fp16.h>

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
  asm volatile("griddepcontrol.launch_dependents;");  // the merge grid may be scheduled now
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

// ---------------------------------------------------------------------------
// Tensor-core decode for D = 128.  Per item (b, g, 128-position slice):
//   S^T = K Q^T  : M = 128 positions, N = 16 head columns, K = 128 dims
//   O^T = V^T P^T: M = 128 dims,      N = 16 head columns, K = 128 positions
// so an item is 16 tcgen05 MMAs instead of thousands of FMAs.  The group's
// G <= 16 heads are the N columns (columns past G are computed and ignored;
// their P rows stay zero).  Persistent: one CTA per SM; the items are dealt
// round-robin, every whole 128-position slice first and the partial last
// slices of the rows after them, so the CTAs end with the short items and
// stream nearly the same number of bytes.  An item loads only the 32-row TMA
// boxes that hold its positions.  Warp 0 streams K and q with TMA through
// one 3-stage ring and warp 10 streams V through another (K is freed as soon
// as the scores are formed, so more of the next items' bytes are in flight
// while the softmax runs), warp 1 issues the MMAs, and two softmax groups
// (warps 2-5 and 6-9; one thread per position for the scores, per dim for the
// output) take alternate items, so one group's reductions overlap the other's.
// S, O (TMEM), P (shared memory) and the group barriers are indexed by item
// parity.
// ---------------------------------------------------------------------------
// INT8: the cache holds int8 vectors with one fp32 scale per (b, g,
// position).  TMA stages each item's int8 K (with the bf16 q rows) and int8
// V; eight converter warps turn them into fp16 (int8 is exact in fp16, so the
// conversion is exact and needs no multiply) and the MMAs run as fp16 x fp16
// -> fp32.  K goes straight into TMEM as the A operand of the scores (thread
// = position = TMEM lane, 64 columns of fp16 pairs per item), so only V and
// q take fp16 tiles in shared memory, and what that saves buys deeper int8
// staging (three K and three V stages): the staged bytes are what is in flight
// from HBM.  The scales are folded in by the softmax threads, one position
// each: the key scale into the scores, the value scale into P; each thread
// fetches its position's scales one item ahead with cp.async into a small
// ring of its own.
template <bool INT8>
struct TcCfg {
  static constexpr int D = 128;
  static constexpr int NH = 16;                 // head columns of the MMAs
  static constexpr int ROWS = kDecodeSplit;     // positions per item
  static constexpr int NK = 3;                  // K (+q) stages: freed once the scores are formed (int8: K in TMEM)
  static constexpr int NV = INT8 ? 2 : 3;       // V stages: freed once the output is formed
  static constexpr int NSK = 3, NSV = 3;        // int8 staging stages of K (+ bf16 q) and of V
  static constexpr int K_BYTES = INT8 ? 0 : ROWS * D * 2;  // two 64-column boxes (int8: none, K is in TMEM)
  static constexpr int V_BYTES = ROWS * D * 2;
  static constexpr int Q_BYTES = NH * D * 2;    // two boxes of 16 rows
  static constexpr int KSTAGE = K_BYTES + Q_BYTES;
  static constexpr int S8_BYTES = ROWS * D;     // one int8 tile: 128 rows x 128 bytes
  static constexpr int KS_STAGE = S8_BYTES + Q_BYTES;  // int8 K tile + the item's bf16 q rows
  static constexpr int BOX = 32;                // cache rows per TMA box: an item loads ceil(n / 32) boxes
  static constexpr int BOX_BYTES = BOX * 128;   // a box of 128-byte rows (64 bf16 columns or 128 int8 values)
  static constexpr int P_BYTES = NH * ROWS * 2;  // P^T as [head][position], two boxes of 64 positions
  static constexpr int OFF_V = NK * KSTAGE;
  static constexpr int OFF_KS = OFF_V + NV * V_BYTES;                 // int8 K staging
  static constexpr int OFF_VS = OFF_KS + (INT8 ? NSK * KS_STAGE : 0);  // int8 V staging
  static constexpr int OFF_P = OFF_VS + (INT8 ? NSV * S8_BYTES : 0);
  static constexpr int OFF_BAR = OFF_P + 2 * P_BYTES;
  static constexpr int OFF_RED = OFF_BAR + 512;  // per group: float rmax[4][NH], rsum[2][4][NH]
  static constexpr int OFF_SC = OFF_RED + 2 * 3 * 4 * NH * 4;  // int8: per group float [2][key|value][ROWS]
  static constexpr int OFF_MISC = OFF_SC + (INT8 ? 2 * 2 * 2 * ROWS * 4 : 0);
  static constexpr int OFF_LENS = OFF_MISC + 64;
  static constexpr int MAX_B = 1024;             // batch rows staged in shared memory
  static constexpr int OFF_PRE = OFF_LENS + MAX_B * 4;
  static constexpr int SMEM = OFF_PRE + (MAX_B + 1) * 4 + 1024;
  static constexpr int kThreads = INT8 ? 640 : 384;  // + warps 12-15 converting K, 16-19 converting V
  // TMEM: S_b at 16b (b = item parity), O_b at 32 + 16b (b = item mod 4); int8: K stage i at 128 + 64i
  static constexpr int T_O = 32;
  static constexpr int T_K = 128;
  static constexpr int TMEM_COLS = INT8 ? 512 : 128;
  static_assert(!INT8 || T_K + NK * 64 <= TMEM_COLS, "TMEM budget");
  static_assert(KSTAGE % 1024 == 0 && OFF_V % 1024 == 0 && OFF_KS % 1024 == 0 && OFF_VS % 1024 == 0 &&
                    OFF_P % 1024 == 0, "swizzled tiles need 1024-byte alignment");
  static_assert(SMEM <= 232448, "shared memory budget");
  static_assert(ROWS == 128, "one position per softmax / converter thread");
  static_assert(BOX_BYTES % 1024 == 0, "boxes keep the 128-byte swizzle phase");
};
template <int NK, int NV>
struct TcBars {
  uint64_t kfull[NK], kempty[NK], vfull[NV], vempty[NV];
  uint64_t ksfull[4], ksempty[4], vsfull[3], vsempty[3];  // int8 staging
  uint64_t s_full[2], p_full[2], o_full[4];
  uint64_t done, done2;
};
namespace tcd {
constexpr int MAX_B = TcCfg<false>::MAX_B;
}  // namespace tcd

// 16 cached int8 values (one 16-byte chunk) to 8 words of fp16 pairs
// (values 2i, 2i + 1 in word i, the lower index in the low half), exactly:
// the biased byte b = x + 128 in the mantissa of fp16 1024 is 1024 + b, and
// subtracting 1152 leaves x
__device__ __forceinline__ void int8_chunk_to_f16(const uint4 w, uint32_t (&o)[8]) {
  const uint32_t nmagic = 0xE480E480u;  // fp16x2 (-1152, -1152)
  const uint32_t wv[4] = {w.x ^ 0x80808080u, w.y ^ 0x80808080u, w.z ^ 0x80808080u, w.w ^ 0x80808080u};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    // fp16 pairs (1024 + b0, 1024 + b1) and (1024 + b2, 1024 + b3)
    const uint32_t lo = __byte_perm(wv[i], 0x64646464u, 0x5140);
    const uint32_t hi = __byte_perm(wv[i], 0x64646464u, 0x7362);
    uint32_t x;
    asm("add.rn.f16x2 %0, %1, %2;" : "=r"(x) : "r"(lo), "r"(nmagic));
    o[2 * i] = x;
    asm("add.rn.f16x2 %0, %1, %2;" : "=r"(x) : "r"(hi), "r"(nmagic));
    o[2 * i + 1] = x;
  }
}

// one cached int8 row (128 values, staged with a 128-byte swizzle) to fp16
// row r of a K-major, 128-byte-swizzled tile of two 64-column boxes
__device__ __forceinline__ void int8_row_to_f16(const unsigned char* stg, unsigned char* tile, int r) {
#pragma unroll
  for (int c = 0; c < 8; ++c) {  // 16 values per 16-byte chunk
    const uint4 w = *reinterpret_cast<const uint4*>(stg + r * 128 + ((c ^ (r & 7)) << 4));
    uint32_t o[8];
    int8_chunk_to_f16(w, o);
    unsigned char* box = tile + (c >> 2) * (128 * 128) + r * 128;
    const int cc = 2 * (c & 3);
    *reinterpret_cast<uint4*>(box + ((cc ^ (r & 7)) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
    *reinterpret_cast<uint4*>(box + (((cc + 1) ^ (r & 7)) << 4)) = make_uint4(o[4], o[5], o[6], o[7]);
  }
}

// 4-byte asynchronous copy global -> shared (cp.async, completion per thread by group)
__device__ __forceinline__ void cp_async4(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// instruction descriptor, kind::f16 with fp16 A/B and fp32 accumulation
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N, int a_mn_major, int b_mn_major) {
  return (1u << 4) | (uint32_t(a_mn_major) << 15) | (uint32_t(b_mn_major) << 16) | (uint32_t(N >> 3) << 17) |
         (uint32_t(M >> 4) << 24);
}

// Item slot j of the deal: the whole 128-position slices of every row come
// first (pre[b] = whole slices of the rows before b, over all KV heads;
// pre[B] = their count), then one slot per row (b, g) for its partial last
// slice, empty (n == 0) when lens[b] is a multiple of 128.  Dealing the
// whole slices first and the short ones last evens out the bytes per CTA.
struct Item {
  int b, g, sp, len, nsplit, n;  // n: positions of the slice in the cache
};
// Every role visits its slots in increasing j, so the row of a whole slice
// is found by walking on from the previous one (no search per item).
struct ItemWalk {
  int b = 0;
  __device__ __forceinline__ Item at(int j, const int* pre, const int* lens, int B, int Hkv) {
    Item it;
    const int nfull = pre[B];
    if (j < nfull) {
      while (pre[b + 1] <= j) ++b;  // the last row with pre[b] <= j (pre[B] > j ends the walk)
      it.b = b;
      it.len = lens[b];
      const int nf = it.len / kDecodeSplit;
      const int r = j - pre[b];
      it.g = r / nf;
      it.sp = r - it.g * nf;
      it.n = kDecodeSplit;
    } else {
      const int r = j - nfull;
      it.b = r / Hkv;
      it.g = r - it.b * Hkv;
      it.len = lens[it.b];
      it.sp = it.len / kDecodeSplit;
      it.n = it.len - it.sp * kDecodeSplit;
    }
    it.nsplit = (it.len + kDecodeSplit - 1) / kDecodeSplit;
    return it;
  }
};

template <int GMAX, bool INT8>
__global__ void __launch_bounds__(TcCfg<INT8>::kThreads, 1) gqa_decode_tc_kernel(const __grid_constant__ DecodeArgs a,
                                                                                float scale_log2, int max_split) {
  using C = TcCfg<INT8>;
  constexpr int D = C::D, NH = C::NH, ROWS = C::ROWS, NK = C::NK, NV = C::NV, K_BYTES = C::K_BYTES;
  constexpr int KSTAGE = C::KSTAGE, V_BYTES = C::V_BYTES, P_BYTES = C::P_BYTES, OFF_V = C::OFF_V, OFF_P = C::OFF_P;
  constexpr int OFF_BAR = C::OFF_BAR, OFF_RED = C::OFF_RED, OFF_MISC = C::OFF_MISC, OFF_LENS = C::OFF_LENS;
  constexpr int OFF_PRE = C::OFF_PRE, kThreadsTc = C::kThreads;
  using Bars = TcBars<NK, NV>;
  static_assert(sizeof(Bars) <= 512, "barrier space");
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Bars& bar = *reinterpret_cast<Bars*>(smem + OFF_BAR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_MISC + 16);
  int* lens_s = reinterpret_cast<int*>(smem + OFF_LENS);
  int* pre = reinterpret_cast<int*>(smem + OFF_PRE);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = a.Hq / a.Hkv;
  const int ncta = gridDim.x, cta = blockIdx.x;
  const Abort ab{abort_flag, a.err};
  asm volatile("griddepcontrol.launch_dependents;");  // the merge grid may be scheduled now

  // set-up that reads no input overlaps the previous kernel in the stream
  // (this grid is launched as a programmatic dependent)
  if (tid == 0) {
    // int8: a K or V stage completes when its 128 converter threads have written it
    for (int i = 0; i < NK; ++i) { mbar_init(&bar.kfull[i], INT8 ? 128 : 1); mbar_init(&bar.kempty[i], 1); }
    for (int i = 0; i < NV; ++i) { mbar_init(&bar.vfull[i], INT8 ? 128 : 1); mbar_init(&bar.vempty[i], 1); }
    for (int i = 0; i < C::NSK; ++i) { mbar_init(&bar.ksfull[i], 1); mbar_init(&bar.ksempty[i], 128); }
    for (int i = 0; i < C::NSV; ++i) { mbar_init(&bar.vsfull[i], 1); mbar_init(&bar.vsempty[i], 128); }
    for (int i = 0; i < 2; ++i) { mbar_init(&bar.s_full[i], 1); mbar_init(&bar.p_full[i], 128); }
    for (int i = 0; i < 4; ++i) mbar_init(&bar.o_full[i], 1);
    mbar_init(&bar.done, 1);
    mbar_init(&bar.done2, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) { tmem_alloc(tmem_slot, C::TMEM_COLS); tmem_relinquish(); }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&a.tk); prefetch_tmap(&a.tv); prefetch_tmap(&a.tq); prefetch_tmap(&a.tk2); prefetch_tmap(&a.tv2);
  }
  // P rows of heads past G are never written again: zero both P buffers once
  for (int i = tid; i < 2 * P_BYTES / 16; i += kThreadsTc)
    reinterpret_cast<uint4*>(smem + OFF_P)[i] = make_uint4(0, 0, 0, 0);
  asm volatile("griddepcontrol.wait;" ::: "memory");  // inputs written by earlier kernels are visible
  // stage (and validate) the lengths; rows with an empty cache get zeros here
  for (int bb = tid; bb < a.B; bb += kThreadsTc) {
    const int l = a.lens[bb];
    if ((l < 0 || l > a.Smax) && cta == 0) atomicExch(a.err, DEV_LENS_CLAMPED);
    lens_s[bb] = l < 0 ? 0 : (l > a.Smax ? a.Smax : l);
  }
  fence_proxy_async_smem();
  __syncthreads();
  if (warp == 0) {  // exclusive prefix of whole slices per row: each lane scans a run of rows
    const int per = (a.B + 31) / 32, b0 = lane * per, b1 = min(a.B, b0 + per);
    int run = 0;
    for (int bb = b0; bb < b1; ++bb) run += lens_s[bb] / kDecodeSplit * a.Hkv;
    int inc = run;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += t;
    }
    int acc = inc - run;
    for (int bb = b0; bb < b1; ++bb) {
      pre[bb] = acc;
      acc += lens_s[bb] / kDecodeSplit * a.Hkv;
    }
    if (lane == 31) pre[a.B] = inc;
  } else {
    __nv_bfloat16* ob = static_cast<__nv_bfloat16*>(a.out);
    for (int bb = cta; bb < a.B; bb += ncta)
      if (lens_s[bb] == 0)
        for (int x = tid - 32; x < a.Hq * D; x += kThreadsTc - 32) ob[(size_t)bb * a.Hq * D + x] = __float2bfloat16(0.f);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int total = pre[a.B] + a.B * a.Hkv;  // item slots
  const int n_slots = cta < total ? (total - cta + ncta - 1) / ncta : 0;  // this CTA's slots i: j = cta + i*ncta
  // every role walks the same slots and skips the same empty ones, so the
  // item counter k (ring stages, buffers, phases) agrees between them
  auto count_items = [&]() {
    int n = 0;
    ItemWalk w;
    for (int i = 0; i < n_slots; ++i) n += w.at(cta + i * ncta, pre, lens_s, a.B, a.Hkv).n > 0;
    return n;
  };

  if (warp == 0 || warp == 10) {
    // ---------------------------------------------------------- TMA producers: K and q (warp 0), V (warp 10)
    // (int8: into the staging tiles).  An item loads only the 32-row boxes
    // that hold its positions.
    if (lane == 0) {
      const bool is_v = warp == 10;
      int k = 0;
      ItemWalk walk;
      for (int i = 0; i < n_slots; ++i) {
        const Item it = walk.at(cta + i * ncta, pre, lens_s, a.B, a.Hkv);
        if (it.n == 0) continue;
        // a whole slice in one 128-row box per 64 columns, a short one in the
        // 32-row boxes that hold its positions
        const bool whole = it.n == ROWS;
        const int nb = whole ? 1 : (it.n + C::BOX - 1) / C::BOX, t0 = it.sp * ROWS;
        const int bbytes = whole ? ROWS * 128 : C::BOX_BYTES, brows = whole ? ROWS : C::BOX;
        const CUtensorMap* mk = whole ? &a.tk : &a.tk2;
        const CUtensorMap* mv = whole ? &a.tv : &a.tv2;
        if (INT8) {
          const int ns = is_v ? C::NSV : C::NSK;
          const int st = k % ns;
          uint64_t* fb = is_v ? &bar.vsfull[st] : &bar.ksfull[st];
          if (!mbar_wait(is_v ? &bar.vsempty[st] : &bar.ksempty[st], ((k / ns) & 1) ^ 1, ab)) break;
          unsigned char* sb = smem + (is_v ? C::OFF_VS + st * C::S8_BYTES : C::OFF_KS + st * C::KS_STAGE);
          mbar_expect_tx(fb, nb * bbytes + (is_v ? 0 : C::Q_BYTES));
          for (int jb = 0; jb < nb; ++jb)
            tma_load_4d(sb + jb * bbytes, is_v ? mv : mk, fb, 0, t0 + jb * brows, it.g, it.b);
          if (!is_v)
            for (int bx = 0; bx < 2; ++bx)
              tma_load_3d(sb + C::S8_BYTES + bx * (NH * 128), &a.tq, fb, bx * 64, it.g * G, it.b);
        } else {
          const int ns = is_v ? NV : NK;
          const int st = k % ns;
          uint64_t* fb = is_v ? &bar.vfull[st] : &bar.kfull[st];
          if (!mbar_wait(is_v ? &bar.vempty[st] : &bar.kempty[st], ((k / ns) & 1) ^ 1, ab)) break;
          unsigned char* sb = smem + (is_v ? OFF_V + st * V_BYTES : st * KSTAGE);
          mbar_expect_tx(fb, 2 * nb * bbytes + (is_v ? 0 : C::Q_BYTES));
          for (int bx = 0; bx < 2; ++bx) {
            for (int jb = 0; jb < nb; ++jb)
              tma_load_4d(sb + bx * (ROWS * 128) + jb * bbytes, is_v ? mv : mk, fb, bx * 64, t0 + jb * brows, it.g,
                          it.b);
            if (!is_v) tma_load_3d(sb + K_BYTES + bx * (NH * 128), &a.tq, fb, bx * 64, it.g * G, it.b);
          }
        }
        ++k;
      }
    }
  } else if (INT8 && warp >= 12) {
    // ---------------------------------------------------------- int8 -> fp16 converters
    // warps 12-15 convert K into TMEM (thread = position = TMEM lane of its
    // warp's quarter) and the item's q rows (bf16 -> fp16) into shared
    // memory; warps 16-19 convert V, thread r owning row r.  A failed wait
    // runs on (the tiles are then garbage and the error word is set)
    const bool is_v = warp >= 16;
    const int r = is_v ? tid - 512 : (warp & 3) * 32 + lane;
    const int n_items = count_items();
    for (int k = 0; k < n_items; ++k) {
      if (!is_v) {
        const int kst = k % NK, ss = k % C::NSK;
        mbar_wait(&bar.kempty[kst], ((k / NK) & 1) ^ 1, ab);
        mbar_wait(&bar.ksfull[ss], (k / C::NSK) & 1, ab);
        tc_fence_after();
        const unsigned char* sb = smem + C::OFF_KS + ss * C::KS_STAGE;
        unsigned char* kb = smem + kst * KSTAGE;  // the q stage (K itself is in TMEM)
        const uint32_t tk = tmem + (uint32_t((warp & 3) * 32) << 16) + C::T_K + kst * 64;
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {  // dims 64hh .. 64hh + 63: TMEM columns 32hh .. 32hh + 31
          uint32_t o[32];
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const int cg = 4 * hh + c;
            uint32_t w8[8];
            int8_chunk_to_f16(*reinterpret_cast<const uint4*>(sb + r * 128 + ((cg ^ (r & 7)) << 4)), w8);
#pragma unroll
            for (int i = 0; i < 8; ++i) o[8 * c + i] = w8[i];
          }
          tmem_st32(tk + hh * 32, o);
        }
        // q: 16 rows x 128 bf16 in two swizzled boxes; thread r converts 16 values in place order
        {
          const uint4 u0 = reinterpret_cast<const uint4*>(sb + C::S8_BYTES)[2 * r];
          const uint4 u1 = reinterpret_cast<const uint4*>(sb + C::S8_BYTES)[2 * r + 1];
          const uint32_t in[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
          uint32_t o[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            float x0 = bf16lo(in[i]), x1 = bf16hi(in[i]);
            uint32_t h;
            asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(h) : "f"(x1), "f"(x0));
            o[i] = h;
          }
          reinterpret_cast<uint4*>(kb + K_BYTES)[2 * r] = make_uint4(o[0], o[1], o[2], o[3]);
          reinterpret_cast<uint4*>(kb + K_BYTES)[2 * r + 1] = make_uint4(o[4], o[5], o[6], o[7]);
        }
        fence_proxy_async_smem();
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&bar.ksempty[ss]);
        mbar_arrive(&bar.kfull[kst]);
      } else {
        const int vst = k % NV, ss = k % C::NSV;
        mbar_wait(&bar.vempty[vst], ((k / NV) & 1) ^ 1, ab);
        mbar_wait(&bar.vsfull[ss], (k / C::NSV) & 1, ab);
        int8_row_to_f16(smem + C::OFF_VS + ss * C::S8_BYTES, smem + OFF_V + vst * V_BYTES, r);
        fence_proxy_async_smem();
        mbar_arrive(&bar.vsempty[ss]);
        mbar_arrive(&bar.vfull[vst]);
      }
    }
  } else if (warp == 1 || warp == 11) {
    // ---------------------------------------------------------- MMA issuers
    // warp 1 issues the scores, warp 11 the outputs: one thread issues a
    // tcgen05.mma about every 60 cycles whatever its size, and an item's
    // sixteen small MMAs with their commits and waits took one thread longer
    // than the item's bytes take to stream.  The two sequences share no TMEM
    // columns and no shared-memory operand; a group writes P(k+2) only after
    // O(k) has completed, which keeps two P buffers and barriers enough.
    {
      // K (K-major; int8 cache: fp16 in TMEM) x q (K-major); V^T (MN-major) x P^T (K-major); fp16
      // operands for the int8 cache
      constexpr uint32_t IDESC_S = INT8 ? idesc_f16(128, NH, 0, 0) : idesc_bf16(128, NH, 0, 0);
      constexpr uint32_t IDESC_O = INT8 ? idesc_f16(128, NH, 1, 0) : idesc_bf16(128, NH, 1, 0);
      const uint32_t s0 = smem_u32(smem);
      auto issue_s = [&](int k) {
        const uint32_t sb = s0 + (k % NK) * KSTAGE;
        const uint64_t ak = sdesc_sw128(sb, 16, 1024), bq = sdesc_sw128(sb + K_BYTES, 16, 1024);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint64_t bk = bq + (((kk >> 2) * (NH * 128) + (kk & 3) * 32) >> 4);
          if (INT8)  // K from TMEM: fp16 pairs, 8 columns per 16 dims
            mma_ts(tmem + (k & 1) * 16, tmem + C::T_K + (k % NK) * 64 + kk * 8, bk, IDESC_S, kk > 0 ? 1u : 0u);
          else
            mma_ss(tmem + (k & 1) * 16, ak + (((kk >> 2) * (ROWS * 128) + (kk & 3) * 32) >> 4), bk, IDESC_S,
                   kk > 0 ? 1u : 0u);
        }
        mma_commit(&bar.s_full[k & 1]);
        mma_commit(&bar.kempty[k % NK]);
      };
      auto issue_o = [&](int k) {
        const uint32_t sb = s0 + OFF_V + (k % NV) * V_BYTES;
        const uint64_t av = sdesc_sw128(sb, ROWS * 128, 1024);
        const uint64_t bp = sdesc_sw128(s0 + OFF_P + (k & 1) * P_BYTES, 16, 1024);
#pragma unroll
        for (int kk = 0; kk < ROWS / 16; ++kk)
          mma_ss(tmem + C::T_O + (k & 3) * 16, av + ((kk * 16 * 128) >> 4),
                 bp + (((kk >> 2) * (NH * 128) + (kk & 3) * 32) >> 4), IDESC_O, kk > 0 ? 1u : 0u);
        mma_commit(&bar.o_full[k & 3]);
        mma_commit(&bar.vempty[k % NV]);
      };
      bool ok = true;
      if (warp == 1) {
        if (lane == 0) {
          const int n_items = count_items();
          for (int k = 0; ok && k < n_items; ++k) {
            // S(k) overwrites S(k-2), which its group has read once it has written P(k-2)
            if (k >= 2 && !(ok = mbar_wait(&bar.p_full[k & 1], ((k - 2) >> 1) & 1, ab))) break;
            if (!(ok = mbar_wait(&bar.kfull[k % NK], (k / NK) & 1, ab))) break;
            tc_fence_after();
            issue_s(k);
          }
          mma_drain(&bar.done, a.err);
        }
      } else {
        // the whole warp waits for each V tile in turn (never more than one
        // phase behind its barrier: the next tile of a stage lands only after
        // this warp's O of the current one) and, for a partial slice, zeroes
        // the value rows at or past the length before O reads them: they were
        // loaded from a cache that may hold anything there, or not loaded and
        // left by an earlier item (or never written), and get zero weight
        ItemWalk walk;
        int k = 0;
        for (int i = 0; ok && i < n_slots; ++i) {
          const Item it = walk.at(cta + i * ncta, pre, lens_s, a.B, a.Hkv);
          if (it.n == 0) continue;
          ok = __all_sync(0xffffffffu, mbar_wait(&bar.vfull[k % NV], (k / NV) & 1, ab));
          if (!ok) break;
          if (!INT8 && it.n < ROWS) {
            unsigned char* vb = smem + OFF_V + (k % NV) * V_BYTES;
            for (int x = lane; x < (ROWS - it.n) * 16; x += 32) {  // 16-byte chunks: 8 per row in each of two boxes
              const int row = it.n + (x >> 4), c = x & 15;
              *reinterpret_cast<uint4*>(vb + (c >> 3) * (ROWS * 128) + row * 128 + (c & 7) * 16) = make_uint4(0, 0, 0, 0);
            }
            fence_proxy_async_smem();
            __syncwarp();
          }
          if (lane == 0) {
            ok = mbar_wait(&bar.p_full[k & 1], (k >> 1) & 1, ab);
            if (ok) {
              tc_fence_after();
              issue_o(k);
            }
          }
          ok = __shfl_sync(0xffffffffu, ok, 0);
          ++k;
        }
        if (lane == 0) mma_drain(&bar.done2, a.err);
      }
    }
  } else {
    // ---------------------------------------------------------- softmax + epilogue
    // group gi takes items k = gi, gi + 2, ...; thread = TMEM lane = position
    // (scores) and = dim (output); control flow is uniform over the group's
    // 128 threads, so its named barrier completes.  An item's output is read
    // after the group has written the next item's P (which waits for that
    // output, as it reuses its P buffer), so the tensor core forms O while the
    // group already works on the next scores (O in TMEM and its barriers by
    // k & 3).  rmax is rewritten only once the group's next scores
    // exist, which needs every thread's P of this item; an item's rsum (by
    // item parity within the group) is read after the next item's barrier and
    // rewritten only after the barrier of the item after that.
    const int gi = (warp - 2) >> 2;
    const int wq = warp & 3;            // TMEM lane quarter of this warp
    const int r = wq * 32 + lane;       // position / dim handled by this thread
    const uint32_t lane_base = uint32_t(wq * 32) << 16;
    float* rmax = reinterpret_cast<float*>(smem + OFF_RED) + gi * 3 * 4 * NH;
    float* rsum0 = rmax + 4 * NH;
    __nv_bfloat16* ogb = static_cast<__nv_bfloat16*>(a.out);
    // this group's items in order (k counts the CTA's non-empty slots)
    ItemWalk walk;
    int ni = 0, nk = -1;
    auto next_mine = [&](Item& nit, int& kk) {
      for (; ni < n_slots; ++ni) {
        nit = walk.at(cta + ni * ncta, pre, lens_s, a.B, a.Hkv);
        if (nit.n == 0) continue;
        if ((++nk & 1) != gi) continue;
        kk = nk;
        ++ni;
        return true;
      }
      return false;
    };
    // int8 cache: position r's key and value scales, fetched one item ahead
    // into this thread's slots of a two-item ring (a cold load, or a register
    // carried over from a load issued one item earlier, would otherwise sit on
    // every item's path).  One copy group per item, empty where the item has
    // no position r or there is no next item, so that waiting for all but the
    // newest group always covers the current item.
    float* scr = reinterpret_cast<float*>(smem + C::OFF_SC) + gi * 2 * 2 * ROWS + r;
    auto fetch_scales = [&](const Item& sit, int kk, bool any) {
      if (!INT8) return;
      if (any && r < sit.n) {  // positions past the length are never read (p is 0 there)
        const size_t so = ((size_t)sit.b * a.Hkv + sit.g) * a.Smax + sit.sp * ROWS + r;
        float* d = scr + ((kk >> 1) & 1) * 2 * ROWS;
        cp_async4(d, a.kscale + so);
        cp_async4(d + ROWS, a.vscale + so);
      }
      cp_async_commit();
    };
    // the output of item (pit, pk): thread r owns dim r of every head
    auto wait_o = [&](int pk) {
      mbar_wait(&bar.o_full[pk & 3], (pk >> 2) & 1, ab);
      tc_fence_after();
    };
    auto epilogue = [&](const Item& pit, int pk) {
      const float* rs = rsum0 + ((pk >> 1) & 1) * 4 * NH;
      uint32_t orr[16];
      tmem_ld16(tmem + lane_base + C::T_O + (pk & 3) * 16, orr);
      tmem_ld_wait();
      __nv_bfloat16* og = ogb + ((size_t)pit.b * a.Hq + (size_t)pit.g * G) * D;
      const int bg = pit.b * a.Hkv + pit.g;
#pragma unroll
      for (int h = 0; h < GMAX; ++h) {
        if (h >= G) continue;
        const float L = (rs[h] + rs[NH + h]) + (rs[2 * NH + h] + rs[3 * NH + h]);
        const float o = __uint_as_float(orr[h]);
        if (pit.nsplit == 1) {
          og[h * D + r] = __float2bfloat16(o / L);
        } else {
          a.part_o[(((size_t)bg * max_split + pit.sp) * GMAX + h) * D + r] = o;
          if (r == 0) a.part_ml[(((size_t)bg * max_split + pit.sp) * GMAX + h) * 2 + 1] = L;
        }
      }
    };
    Item it, pit;
    int k = 0, pk = 0;
    bool have = next_mine(it, k), have_prev = false;
    fetch_scales(it, k, have);
    while (have) {
      Item itn;
      int kn = 0;
      const bool have_n = next_mine(itn, kn);
      fetch_scales(itn, kn, have_n);
      const int buf = k & 1;
      const uint32_t par = (k >> 1) & 1;
      const int n = it.n;
      float ksc = 1.f, vsc = 1.f;
      if (INT8 && r < n) {
        cp_async_wait<1>();  // this item's copies (the newest group is the next item's)
        ksc = scr[par * 2 * ROWS];
        vsc = scr[par * 2 * ROWS + ROWS];
      }
      // a failed wait (abort or timeout) runs on: the named barriers need every thread
      mbar_wait(&bar.s_full[buf], par, ab);
      tc_fence_after();
      uint32_t sr[16];
      tmem_ld16(tmem + lane_base + buf * 16, sr);
      tmem_ld_wait();
      float sv[GMAX];
#pragma unroll
      for (int h = 0; h < GMAX; ++h)
        sv[h] = (h < G && r < n) ? __uint_as_float(sr[h]) * (scale_log2 * ksc) : -INFINITY;
      // max over the item's positions, per head
#pragma unroll
      for (int h = 0; h < GMAX; ++h) {
        float m = sv[h];
#pragma unroll
        for (int off = 16; off; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
        if (lane == 0) rmax[wq * NH + h] = m;
      }
      named_bar(1 + gi, 128);
      float p[GMAX];
#pragma unroll
      for (int h = 0; h < GMAX; ++h) {
        const float M = fmaxf(fmaxf(rmax[h], rmax[NH + h]), fmaxf(rmax[2 * NH + h], rmax[3 * NH + h]));
        p[h] = (h < G && r < n) ? fast_exp2(sv[h] - M) : 0.f;
        if (h < G && r == 0 && it.nsplit > 1)
          a.part_ml[(((size_t)(it.b * a.Hkv + it.g) * max_split + it.sp) * GMAX + h) * 2] = M;
      }
      // P^T[head][position] in the K-major 128-byte-swizzled layout of the MMA's B operand,
      // once O of the group's previous item has read the buffer
      if (have_prev) wait_o(pk);
      {
        unsigned char* pb = smem + OFF_P + buf * P_BYTES + (r >> 6) * (NH * 128);
        const int chunk = (r & 63) >> 3;
#pragma unroll
        for (int h = 0; h < GMAX; ++h)
          if (h < G) {
            unsigned short* dst = reinterpret_cast<unsigned short*>(pb + h * 128 + ((chunk ^ (h & 7)) << 4) + (r & 7) * 2);
            if (INT8)
              *dst = __half_as_ushort(__float2half_rn(p[h] * vsc));  // value scale folded into P (fp16)
            else
              *dst = __bfloat16_as_ushort(__float2bfloat16(p[h]));
          }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&bar.p_full[buf]);
      // the denominators while the tensor core forms O
      float* rs = rsum0 + par * 4 * NH;
#pragma unroll
      for (int h = 0; h < GMAX; ++h) {
        float l = p[h];
#pragma unroll
        for (int off = 16; off; off >>= 1) l += __shfl_xor_sync(0xffffffffu, l, off);
        if (lane == 0) rs[wq * NH + h] = l;
      }
      // the previous item's output (its sums were complete at this item's barrier)
      if (have_prev) epilogue(pit, pk);
      pit = it;
      pk = k;
      have_prev = true;
      it = itn;
      k = kn;
      have = have_n;
    }
    if (have_prev) {
      named_bar(1 + gi, 128);  // every warp's sums of the last item
      wait_o(pk);
      epilogue(pit, pk);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// merge the slices of every row (b, g) that has more than one: one CTA of D
// threads per (b, g, head h), thread = dim; each thread loads the (max, sum,
// partial) of sixteen slices at a time, all in flight together, merging
// chunks of slices online (a chain of dependent global loads here would cost
// more than the attention itself).  The CTAs are small, so they can be
// resident beside the attention grid's and start as soon as it completes.
template <int D, int GMAX>
__global__ void __launch_bounds__(D) gqa_decode_combine_kernel(DecodeArgs a, int max_split) {
  const int G = a.Hq / a.Hkv;
  const int bg = blockIdx.x / G, h = blockIdx.x - bg * G;
  const int b = bg / a.Hkv, g = bg - b * a.Hkv, d = threadIdx.x;
  // launched early (programmatic dependent launch): the partials are
  // complete and visible once the attention grid has finished, and so is
  // every input written before it (the attention grid itself waits for its
  // predecessors), so lens is read only after the wait; the next kernel in
  // the stream may then start its own set-up
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");
  int len = a.lens[b];
  len = len < 0 ? 0 : (len > a.Smax ? a.Smax : len);
  const int nsplit = (len + kDecodeSplit - 1) / kDecodeSplit;
  if (nsplit <= 1) return;
  const float* ml0 = a.part_ml + ((size_t)bg * max_split * GMAX + h) * 2;
  const float* po = a.part_o + ((size_t)bg * max_split * GMAX + h) * D + d;
  float M = -INFINITY, L = 0.f, acc = 0.f;
  for (int s0 = 0; s0 < nsplit; s0 += 16) {
    float o[16], m[16], l[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const bool in = s0 + j < nsplit;
      const float* ml = ml0 + (size_t)(s0 + j) * GMAX * 2;
      o[j] = in ? po[(size_t)(s0 + j) * GMAX * D] : 0.f;
      m[j] = in ? ml[0] : -INFINITY;
      l[j] = in ? ml[1] : 0.f;
    }
    float mc = m[0];
#pragma unroll
    for (int j = 1; j < 16; ++j) mc = fmaxf(mc, m[j]);
    const float mn = fmaxf(M, mc);  // finite: every chunk holds at least one slice
    const float f = fast_exp2(M - mn);
    acc *= f;
    L *= f;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const float w = fast_exp2(m[j] - mn);  // 0 for slices past nsplit
      acc = fmaf(o[j], w, acc);
      L = fmaf(l[j], w, L);
    }
    M = mn;
  }
  static_cast<__nv_bfloat16*>(a.out)[((size_t)b * a.Hq + (size_t)g * G + h) * D + d] = __float2bfloat16(acc / L);
}

// the merge grid may be scheduled while the attention grid still runs (its
// CTAs are small and wait in griddepcontrol.wait), hiding its launch latency
template <int D, int GMAX>
cudaError_t launch_combine(const DecodeArgs& a, int max_split, cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.B * a.Hkv * (a.Hq / a.Hkv));
  cfg.blockDim = dim3(D);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, gqa_decode_combine_kernel<D, GMAX>, a, max_split);
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
  return max_split > 1 ? launch_combine<D, GMAX>(a, max_split, st) : cudaSuccess;
}

template <int GMAX, bool INT8>
cudaError_t launch_tc(const DecodeArgs& a0, cudaStream_t st) {
  using C = TcCfg<INT8>;
  DecodeArgs a = a0;
  const unsigned long long D = 128, eb = INT8 ? 1 : 2;  // bytes per cached element
  unsigned long long kd[4] = {D, (unsigned long long)a.Smax, (unsigned long long)a.Hkv, (unsigned long long)a.B};
  unsigned long long ks[3] = {D * eb, (unsigned long long)a.Smax * D * eb, (unsigned long long)a.Hkv * a.Smax * D * eb};
  unsigned kb[4] = {INT8 ? 128u : 64u, (unsigned)C::ROWS, 1, 1};  // 128-byte rows either way
  unsigned kb2[4] = {INT8 ? 128u : 64u, (unsigned)C::BOX, 1, 1};  // short slices
  unsigned long long qd[3] = {D, (unsigned long long)a.Hq, (unsigned long long)a.B};
  unsigned long long qs[2] = {D * 2, (unsigned long long)a.Hq * D * 2};
  unsigned qb[3] = {64, (unsigned)C::NH, 1};
  if (encode_tmap(&a.tk, a.kc, 4, kd, ks, kb, (int)eb) || encode_tmap(&a.tv, a.vc, 4, kd, ks, kb, (int)eb) ||
      encode_tmap(&a.tk2, a.kc, 4, kd, ks, kb2, (int)eb) || encode_tmap(&a.tv2, a.vc, 4, kd, ks, kb2, (int)eb) ||
      encode_tmap(&a.tq, a.q, 3, qd, qs, qb, 2))
    return cudaErrorInvalidValue;
  auto kern = gqa_decode_tc_kernel<GMAX, INT8>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int max_split = decode_max_split(a.Smax);
  const float scale_log2 = 1.4426950408889634f / sqrtf((float)a.D);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(sms);
  cfg.blockDim = dim3(C::kThreads);
  cfg.dynamicSmemBytes = C::SMEM;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // its set-up overlaps the previous kernel
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if ((e = cudaLaunchKernelEx(&cfg, kern, a, scale_log2, max_split)) != cudaSuccess) return e;
  return max_split > 1 ? launch_combine<128, GMAX>(a, max_split, st) : cudaSuccess;
}

template <bool INT8>
cudaError_t launch_tc_g(const DecodeArgs& a, cudaStream_t st) {
  const int G = a.Hq / a.Hkv;
  if (G <= 1) return launch_tc<1, INT8>(a, st);
  if (G <= 2) return launch_tc<2, INT8>(a, st);
  if (G <= 4) return launch_tc<4, INT8>(a, st);
  if (G <= 8) return launch_tc<8, INT8>(a, st);
  return launch_tc<16, INT8>(a, st);
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

int decode_max_split(int Smax) { return (int)(((long long)Smax + kDecodeSplit - 1) / kDecodeSplit); }

static int gmax_of(int G) { return G <= 1 ? 1 : G <= 2 ? 2 : G <= 4 ? 4 : G <= 8 ? 8 : 16; }

size_t decode_part_o_floats(int B, int Hq, int Hkv, int Smax, int D) {
  return (size_t)B * Hkv * decode_max_split(Smax) * gmax_of(Hq / Hkv) * D;
}
size_t decode_part_ml_floats(int B, int Hq, int Hkv, int Smax) {
  return (size_t)B * Hkv * decode_max_split(Smax) * gmax_of(Hq / Hkv) * 2;
}

cudaError_t launch_gqa_decode(const DecodeArgs& a, cudaStream_t st) {
  if (a.kscale) return launch_tc_g<true>(a, st);  // int8 cache (D = 128, B <= 1024 checked by the caller)
  if (a.D == 128 && a.B <= tcd::MAX_B) return launch_tc_g<false>(a, st);  // tensor-core path
  if (a.D == 128) return launch_d<128>(a, st);
  return launch_d<64>(a, st);
}

int decode_int8_max_batch() { return tcd::MAX_B; }

// ---------------------------------------------------------------------------
// Decode without any allocation by the library.
//
// Some callers cannot let a library call cudaMalloc: code running under an
// allocator that owns all device memory (a caching allocator or a memory pool
// sized up front), real-time serving loops that must not hit the driver's
// allocation path or its implicit synchronisation, and processes that have
// reserved nearly all of HBM for the KV cache.  For them the split partials
// of the decode and its error word live in this fixed, statically sized
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

// Read the array's error word (and clear it) on the current device, with
// plain symbol copies that allocate nothing; 0 if the array was never used
// there.  The caller has synchronised the stream the calls ran on.
cudaError_t noalloc_take_error(int* word) {
  *word = 0;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  {
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) return cudaSuccess;
  }
  if ((e = cudaMemcpyFromSymbol(word, cpattn_noalloc_scratch, sizeof(int), 0, cudaMemcpyDeviceToHost)) != cudaSuccess)
    return e;
  if (*word != 0) {
    const int zero = 0;
    e = cudaMemcpyToSymbol(cpattn_noalloc_scratch, &zero, sizeof(int), 0, cudaMemcpyHostToDevice);
  }
  return e;
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
  // every slice partial the merge reads is written by the same call, so
  // nothing left in the array by an earlier call is ever read
  DecodeArgs a{};
  a.q = q; a.kc = kc; a.vc = vc; a.lens = lens; a.out = out;
  a.B = B; a.Hq = Hq; a.Hkv = Hkv; a.Smax = Smax; a.D = D;
  a.part_o = po; a.part_ml = ml; a.err = reinterpret_cast<int*>(base);
  return launch_gqa_decode(a, st);
}

}  // namespace cpattn
