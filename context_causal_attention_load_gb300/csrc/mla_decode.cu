// Absorbed-MLA decode on tcgen05 tensor cores.
//
// MLA attention under context parallelism ("Add support for EP to context
// parallelism in self-attention", Main code changes) at decode time: one new
// query token per sequence against the cache ("Add Pallas GPU decode
// attention in Maxtext inference", Description).  In the absorbed form every
// query head reads the same cached latent row per token, 576 columns: the
// 512-column compressed KV followed by the 64-column rope key.  The row is
// the key of every head, and its first 512 columns are the value:
//   out[b, h] = sum_{t < lens[b]} softmax_t(scale q[b, h] . ckv[b, t]) ckv[b, t, :512].
//
// Work item = (sequence b, chunk of 256 positions), with the heads as the
// MMA rows:
//   S = Q K^T   M = 128 heads, N = 256 positions, K = 576 (nine 64-column boxes)
//   O = P V     M = 128 heads, N = 8 x 64 value columns, K = 256 positions
// TMEM: S in columns [0, 256); after the softmax has read it, O's value
// columns 256-511 go there and columns 0-255 go to [256, 512).  Each item
// writes its partial (o, row max, row sum); a second kernel merges the chunks
// of each (b, h).  Persistent grid, one CTA per SM: the whole chunks of all
// sequences are numbered first and the partial last chunks after them, and
// items are dealt round-robin, so with about one item per SM the short
// chunks are the ones that share an SM.
//
// Roles (192 threads): warps 0-3 softmax and epilogue (thread = head row =
// TMEM lane), warp 4 TMA producer, warp 5 MMA issuer.  One ring of three
// 48 KB stages carries, per item, nine (Q box, K box) pairs for S and then
// the eight value boxes (the first 512 columns of the same rows, now from
// L2).  Positions of a last chunk at or past lens[b] get zero weight; their
// value rows are zeroed in shared memory before O reads them, so whatever
// the cache holds there cannot reach the output.
#include "common.cuh"
#include "internal.h"

namespace cpattn {
namespace {

constexpr int kMdThreads = 192;
constexpr int kMdDk = 576, kMdDv = 512;
constexpr int kMdRows = 128;               // heads per MMA (rows past H are zero)
constexpr int kMdT = 256;                  // positions per chunk
constexpr int kMdKBoxes = kMdDk / 64;      // 9
constexpr int kMdVBoxes = kMdDv / 64;      // 8
constexpr int kMdStagesPerItem = kMdKBoxes + kMdVBoxes;
constexpr int kMdNS = 3;
constexpr int kMdQBox = kMdRows * 128;   // 16 KB
constexpr int kMdKBox = kMdT * 128;      // 32 KB
constexpr int kMdStage = kMdQBox + kMdKBox;
constexpr int kMdOffP = kMdNS * kMdStage;          // P: 4 boxes of 64 positions x 128 rows
constexpr int kMdPBytes = 4 * kMdRows * 128;       // 64 KB
constexpr int kMdOffBar = kMdOffP + kMdPBytes;
constexpr int kMdOffMisc = kMdOffBar + 256;
constexpr int kMdMaxB = 1024;
constexpr int kMdOffLens = kMdOffMisc + 64;
constexpr int kMdOffPre = kMdOffLens + kMdMaxB * 4;            // whole chunks before each sequence
constexpr int kMdOffPre2 = kMdOffPre + (kMdMaxB + 1) * 4;       // partial chunks before each sequence
constexpr int kMdSmem = kMdOffPre2 + (kMdMaxB + 1) * 4 + 1024;
static_assert(kMdSmem <= 232448, "shared memory budget");
static_assert(kMdStage % 1024 == 0 && kMdOffP % 1024 == 0, "swizzled tiles need 1024-byte alignment");

struct MdBars {
  uint64_t full[kMdNS], empty[kMdNS];
  uint64_t s_full, p_full, o_full, o_free;
  uint64_t vfix[kMdVBoxes];
  uint64_t done;
};
static_assert(sizeof(MdBars) <= 256, "barrier area");

struct MdItem {
  int b, chunk, len;
};
// largest b in [0, B) with pre[b] <= j
__device__ __forceinline__ int md_search(int j, const int* pre, int B) {
  int lo = 0, hi = B - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (pre[mid] <= j) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}
// dense item j -> (b, chunk): whole chunks first (pre_full[b] = whole chunks
// of the sequences before b, pre_full[B] their total), then the partial last
// chunks (pre_part[b] = sequences before b that end inside a chunk)
__device__ __forceinline__ MdItem md_item(int j, const int* pre_full, const int* pre_part, const int* lens, int B) {
  const int nfull = pre_full[B];
  if (j < nfull) {
    const int b = md_search(j, pre_full, B);
    return MdItem{b, j - pre_full[b], lens[b]};
  }
  const int b = md_search(j - nfull, pre_part, B);
  return MdItem{b, lens[b] / kMdT, lens[b]};
}

// exclusive prefix over the sequences of f(b) by one warp (each lane scans a
// run of sequences); out[B] receives the total
template <typename F>
__device__ __forceinline__ void md_prefix(int B, int lane, int* out, F f) {
  const int per = (B + 31) / 32, b0 = lane * per, b1 = min(B, b0 + per);
  int run = 0;
  for (int bb = b0; bb < b1; ++bb) run += f(bb);
  int inc = run;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += t;
  }
  int acc = inc - run;
  for (int bb = b0; bb < b1; ++bb) {
    out[bb] = acc;
    acc += f(bb);
  }
  if (lane == 31) out[B] = inc;
}

// TMA store of a tile from shared memory into global memory, tracked by the
// issuing thread's bulk async-group
__device__ __forceinline__ void md_tma_store_4d(const void* src, const CUtensorMap* map, int c0, int c1, int c2, int c3) {
  asm volatile("cp.async.bulk.tensor.4d.global.shared::cta.bulk_group [%0, {%2, %3, %4, %5}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(smem_u32(src)), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
               : "memory");
}
// this thread's bulk async-groups, all but the newest N, have read their sources
template <int N>
__device__ __forceinline__ void md_bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

__global__ void __launch_bounds__(kMdThreads, 1) mla_decode_kernel(const __grid_constant__ MlaDecodeArgs a) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  MdBars& bar = *reinterpret_cast<MdBars*>(smem + kMdOffBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kMdOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kMdOffMisc + 16);
  int* lens_s = reinterpret_cast<int*>(smem + kMdOffLens);
  int* pre = reinterpret_cast<int*>(smem + kMdOffPre);
  int* pre2 = reinterpret_cast<int*>(smem + kMdOffPre2);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int ncta = gridDim.x, cta = blockIdx.x;
  const Abort ab{abort_flag, a.err};
  // the merge grid (a programmatic dependent) may be scheduled now; it waits
  // for this grid before it reads anything
  asm volatile("griddepcontrol.launch_dependents;");

  if (tid == 0) {
    for (int i = 0; i < kMdNS; ++i) { mbar_init(&bar.full[i], 1); mbar_init(&bar.empty[i], 1); }
    mbar_init(&bar.s_full, 1);
    mbar_init(&bar.p_full, 128);
    mbar_init(&bar.o_full, 1);
    mbar_init(&bar.o_free, 128);
    for (int i = 0; i < kMdVBoxes; ++i) mbar_init(&bar.vfix[i], 128);
    mbar_init(&bar.done, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 5) { tmem_alloc(tmem_slot, 512); tmem_relinquish(); }
  if (warp == 4 && lane == 0) { prefetch_tmap(&a.tq); prefetch_tmap(&a.tk); }
  // stage (and validate) the lengths, then number the items
  for (int bb = tid; bb < a.B; bb += kMdThreads) {
    const int l = a.lens[bb];
    if ((l < 0 || l > a.Smax) && cta == 0) atomicExch(a.err, DEV_LENS_CLAMPED);
    lens_s[bb] = l < 0 ? 0 : (l > a.Smax ? a.Smax : l);
  }
  __syncthreads();
  if (warp == 0) md_prefix(a.B, lane, pre, [&](int bb) { return lens_s[bb] / kMdT; });
  if (warp == 1) md_prefix(a.B, lane, pre2, [&](int bb) { return lens_s[bb] % kMdT ? 1 : 0; });
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int total = pre[a.B] + pre2[a.B];
  const int n_items = cta < total ? (total - cta + ncta - 1) / ncta : 0;  // items j = cta + k * ncta

  if (warp == 4) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int g = 0;  // ring stage counter
      bool ok = true;
      for (int k = 0; k < n_items && ok; ++k) {
        const MdItem it = md_item(cta + k * ncta, pre, pre2, lens_s, a.B);
        for (int s = 0; s < kMdStagesPerItem; ++s, ++g) {
          const int st = g % kMdNS;
          if (!(ok = mbar_wait(&bar.empty[st], ((g / kMdNS) & 1) ^ 1, ab))) break;
          unsigned char* sb = smem + st * kMdStage;
          if (s < kMdKBoxes) {  // query box and key box s
            mbar_expect_tx(&bar.full[st], kMdStage);
            tma_load_3d(sb, &a.tq, &bar.full[st], s * 64, 0, it.b);
            tma_load_3d(sb + kMdQBox, &a.tk, &bar.full[st], s * 64, it.chunk * kMdT, it.b);
          } else {  // value box, in the key slot
            const int vb = s - kMdKBoxes;
            mbar_expect_tx(&bar.full[st], kMdKBox);
            tma_load_3d(sb + kMdQBox, &a.tk, &bar.full[st], vb * 64, it.chunk * kMdT, it.b);
          }
        }
      }
      if (!ok) {  // let the copies already issued land (each wait bounded on its own)
        for (int h = g - 1; h >= 0 && h >= g - kMdNS; --h) {
          volatile int own = 0;
          mbar_wait(&bar.full[h % kMdNS], (h / kMdNS) & 1, Abort{&own, a.err});
        }
      }
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t IDESC_S = idesc_bf16(kMdRows, kMdT, 0, 0);  // Q (K-major) x K (K-major)
      constexpr uint32_t IDESC_O = idesc_bf16(kMdRows, 64, 0, 1);    // P (K-major) x V (MN-major)
      const uint32_t s0 = smem_u32(smem);
      const uint64_t pdesc = sdesc_sw128(s0 + kMdOffP, 16, 1024);
      int g = 0, nfix = 0;
      bool ok = true;
      for (int k = 0; k < n_items && ok; ++k) {
        const MdItem it = md_item(cta + k * ncta, pre, pre2, lens_s, a.B);
        const bool partial = it.len - it.chunk * kMdT < kMdT;
        if (k > 0 && !(ok = mbar_wait(&bar.o_free, (k - 1) & 1, ab))) break;  // the last O read out
        for (int c = 0; c < kMdKBoxes; ++c, ++g) {
          const int st = g % kMdNS;
          if (!(ok = mbar_wait(&bar.full[st], (g / kMdNS) & 1, ab))) break;
          tc_fence_after();
          const uint64_t qd = sdesc_sw128(s0 + st * kMdStage, 16, 1024);
          const uint64_t kd = sdesc_sw128(s0 + st * kMdStage + kMdQBox, 16, 1024);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_ss(tmem, qd + ((kk * 32) >> 4), kd + ((kk * 32) >> 4), IDESC_S, (c > 0 || kk > 0) ? 1u : 0u);
          mma_commit(&bar.empty[st]);
        }
        if (!ok) break;
        mma_commit(&bar.s_full);
        if (!(ok = mbar_wait(&bar.p_full, k & 1, ab))) break;  // P written, S read: its columns take O
        tc_fence_after();
        for (int i = 0; i < kMdVBoxes; ++i, ++g) {
          const int st = g % kMdNS;
          if (!(ok = mbar_wait(&bar.full[st], (g / kMdNS) & 1, ab))) break;
          if (partial && !(ok = mbar_wait(&bar.vfix[i], nfix & 1, ab))) break;  // rows past the length zeroed
          tc_fence_after();
          const uint64_t vd = sdesc_sw128(s0 + st * kMdStage + kMdQBox, kMdKBox, 1024);
#pragma unroll
          for (int kk = 0; kk < kMdT / 16; ++kk)
            mma_ss(tmem + (i < 4 ? 256 + 64 * i : 64 * (i - 4)), pdesc + ((((kk >> 2) * (kMdRows * 128)) + (kk & 3) * 32) >> 4),
                   vd + ((kk * 16 * 128) >> 4), IDESC_O, kk > 0 ? 1u : 0u);
          mma_commit(&bar.empty[st]);
        }
        if (!ok) break;
        if (partial) ++nfix;
        mma_commit(&bar.o_full);
      }
      mma_drain(&bar.done, a.err);
    }
  } else if (warp < 4) {
    // ------------------------------------------------------------ softmax and epilogue
    // thread r = head row = TMEM lane; a failed wait runs on (every wait is
    // bounded and the barrier counts still complete)
    const int r = warp * 32 + lane;
    const uint32_t lane_base = uint32_t(warp * 32) << 16;
    const float sl2 = a.scale_log2;
    int nfix = 0;
    for (int k = 0; k < n_items; ++k) {
      const MdItem it = md_item(cta + k * ncta, pre, pre2, lens_s, a.B);
      const int nvalid = min(kMdT, it.len - it.chunk * kMdT);  // positions of the chunk inside the cache
      mbar_wait(&bar.s_full, k & 1, ab);
      tc_fence_after();
      float m = -INFINITY;
#pragma unroll 1
      for (int c = 0; c < kMdT / 32; ++c) {
        uint32_t sv[32];
        tmem_ld32(tmem + lane_base + 32 * c, sv);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 32; ++j)
          if (32 * c + j < nvalid) m = fmaxf(m, __uint_as_float(sv[j]));
      }
      const float m2 = m * sl2;  // finite: every item holds at least one position
      float l = 0.f;
#pragma unroll 1
      for (int c = 0; c < kMdT / 32; ++c) {
        uint32_t sv[32];
        tmem_ld32(tmem + lane_base + 32 * c, sv);
        tmem_ld_wait();
        uint32_t pk[16];
#pragma unroll
        for (int j = 0; j < 32; j += 2) {
          const float p0 = 32 * c + j < nvalid ? fast_exp2(__uint_as_float(sv[j]) * sl2 - m2) : 0.f;
          const float p1 = 32 * c + j + 1 < nvalid ? fast_exp2(__uint_as_float(sv[j + 1]) * sl2 - m2) : 0.f;
          l += p0 + p1;
          pk[j >> 1] = pack_bf16(p0, p1);
        }
        // P row r, positions [32c, 32c+32): box c/2, 16-byte chunks 4(c&1)..+3, 128-byte swizzle
        unsigned char* rowp = smem + kMdOffP + (c >> 1) * (kMdRows * 128) + r * 128;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int ch = 4 * (c & 1) + q;
          *reinterpret_cast<uint4*>(rowp + ((ch ^ (r & 7)) << 4)) =
              make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
        }
      }
      tc_fence_before();
      fence_proxy_async_smem();
      mbar_arrive(&bar.p_full);
      if (nvalid < kMdT) {
        // zero the value rows past the length (stage of value box i of item k)
        for (int i = 0; i < kMdVBoxes; ++i) {
          const int g = k * kMdStagesPerItem + kMdKBoxes + i;
          const int st = g % kMdNS;
          mbar_wait(&bar.full[st], (g / kMdNS) & 1, ab);
          unsigned char* vb = smem + st * kMdStage + kMdQBox;
          for (int row = r; row < kMdT; row += 128)
            if (row >= nvalid)
#pragma unroll
              for (int q = 0; q < 8; ++q) *reinterpret_cast<uint4*>(vb + row * 128 + q * 16) = make_uint4(0, 0, 0, 0);
          fence_proxy_async_smem();
          mbar_arrive(&bar.vfix[i]);
        }
        ++nfix;
      }
      // epilogue: this item's partial (o, row max, row sum); value columns
      // 0-255 are in TMEM [256, 512), 256-511 in [0, 256).  o goes out as
      // sixteen fp32 boxes of 32 columns x 128 head rows, staged four at a
      // time in the P buffer (dead once O is complete; 128-byte swizzle) and
      // written by TMA stores, so the 256 KiB leave in whole lines
      mbar_wait(&bar.o_full, k & 1, ab);
      tc_fence_after();
#pragma unroll 1
      for (int c = 0; c < kMdDv / 32; ++c) {
        uint32_t ov[32];
        tmem_ld32(tmem + lane_base + (c < 8 ? 256 + 32 * c : 32 * (c - 8)), ov);
        tmem_ld_wait();
        unsigned char* buf = smem + kMdOffP + (c & 3) * (kMdRows * 128);
        if (c >= 4) {  // the store that last used this buffer has read it
          if (r == 0) md_bulk_wait_read<3>();
          named_bar(1, 128);
        }
        unsigned char* rp = buf + r * 128;
#pragma unroll
        for (int ch = 0; ch < 8; ++ch)
          *reinterpret_cast<uint4*>(rp + ((ch ^ (r & 7)) << 4)) =
              make_uint4(ov[4 * ch], ov[4 * ch + 1], ov[4 * ch + 2], ov[4 * ch + 3]);
        fence_proxy_async_smem();
        named_bar(1, 128);
        if (r == 0) {
          md_tma_store_4d(buf, &a.tpo, 32 * c, 0, it.chunk, it.b);
          bulk_commit_group();
        }
      }
      const size_t prow = ((size_t)it.b * a.nch + it.chunk) * a.H + r;
      if (r < a.H) {
        a.part_ml[2 * prow] = m2;
        a.part_ml[2 * prow + 1] = l;
      }
      tc_fence_before();
      mbar_arrive(&bar.o_free);
      if (r == 0) md_bulk_wait_read<0>();  // the next item may write P
      named_bar(1, 128);
    }
    if (r == 0) bulk_wait_all();  // the partials have landed before the CTA retires
    (void)nfix;
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// merge of the chunks of each (b, h): one CTA of 128 threads per (b, h),
// four value columns per thread; four chunks' loads in flight at a time,
// merged online.  Launched as a programmatic dependent, so lens and the
// partials are read only after the attention grid has completed.
__global__ void __launch_bounds__(128) mla_decode_merge_kernel(const __grid_constant__ MlaDecodeArgs a) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int b = blockIdx.x / a.H, h = blockIdx.x - b * a.H;
  int len = a.lens[b];
  len = len < 0 ? 0 : (len > a.Smax ? a.Smax : len);
  const int nch = (len + kMdT - 1) / kMdT;
  __nv_bfloat16* o = static_cast<__nv_bfloat16*>(a.out) + ((size_t)b * a.H + h) * kMdDv + 4 * threadIdx.x;
  if (nch == 0) {  // empty cache: zeros
    *reinterpret_cast<uint2*>(o) = make_uint2(0u, 0u);
    return;
  }
  float M = -INFINITY, L = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int c0 = 0; c0 < nch; c0 += 4) {
    float m[4], l[4];
    float4 x[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const bool in = c0 + j < nch;
      const size_t prow = ((size_t)b * a.nch + c0 + j) * a.H + h;
      m[j] = in ? __ldcg(a.part_ml + 2 * prow) : -INFINITY;
      l[j] = in ? __ldcg(a.part_ml + 2 * prow + 1) : 0.f;
      x[j] = in ? __ldcg(reinterpret_cast<const float4*>(a.part_o + prow * kMdDv) + threadIdx.x)
                : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    const float mn = fmaxf(M, fmaxf(fmaxf(m[0], m[1]), fmaxf(m[2], m[3])));  // finite: chunk 0 is in
    const float f = fast_exp2(M - mn);
    L *= f;
    acc.x *= f;
    acc.y *= f;
    acc.z *= f;
    acc.w *= f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float w = fast_exp2(m[j] - mn);  // 0 past the last chunk
      L = fmaf(l[j], w, L);
      acc.x = fmaf(x[j].x, w, acc.x);
      acc.y = fmaf(x[j].y, w, acc.y);
      acc.z = fmaf(x[j].z, w, acc.z);
      acc.w = fmaf(x[j].w, w, acc.w);
    }
    M = mn;
  }
  const float il = 1.f / L;
  *reinterpret_cast<uint2*>(o) = make_uint2(pack_bf16(acc.x * il, acc.y * il), pack_bf16(acc.z * il, acc.w * il));
}

}  // namespace

int mla_decode_chunks(int Smax) { return (int)(((long long)Smax + kMdT - 1) / kMdT); }
int mla_decode_max_batch() { return kMdMaxB; }

cudaError_t launch_mla_decode(const MlaDecodeArgs& a0, int num_sms, cudaStream_t st) {
  MlaDecodeArgs a = a0;
  const unsigned long long Dk = kMdDk;
  unsigned long long qd[3] = {Dk, (unsigned long long)a.H, (unsigned long long)a.B};
  unsigned long long qs[2] = {Dk * 2, (unsigned long long)a.H * Dk * 2};
  unsigned qb[3] = {64, (unsigned)kMdRows, 1};
  unsigned long long kd[3] = {Dk, (unsigned long long)a.Smax, (unsigned long long)a.B};
  unsigned long long ks[2] = {Dk * 2, (unsigned long long)a.Smax * Dk * 2};
  unsigned kb[3] = {64, (unsigned)kMdT, 1};
  unsigned long long pd[4] = {(unsigned long long)kMdDv, (unsigned long long)a.H, (unsigned long long)a.nch,
                              (unsigned long long)a.B};
  unsigned long long ps[3] = {kMdDv * 4ull, (unsigned long long)a.H * kMdDv * 4, (unsigned long long)a.nch * a.H * kMdDv * 4};
  unsigned pb[4] = {32, (unsigned)(a.H < kMdRows ? a.H : kMdRows), 1, 1};
  if (encode_tmap(&a.tq, a.q, 3, qd, qs, qb, 2) || encode_tmap(&a.tk, a.ckv, 3, kd, ks, kb, 2) ||
      encode_tmap(&a.tpo, a.part_o, 4, pd, ps, pb, 4))
    return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(mla_decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kMdSmem);
  if (e != cudaSuccess) return e;
  mla_decode_kernel<<<num_sms, kMdThreads, kMdSmem, st>>>(a);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.B * a.H);
  cfg.blockDim = dim3(128);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, mla_decode_merge_kernel, a);
}

}  // namespace cpattn
