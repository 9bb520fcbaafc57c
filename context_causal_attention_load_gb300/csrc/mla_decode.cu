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
//   O = P V     M = 128 heads, N = 4 x 128 value columns, K = 256 positions
// TMEM: S in columns [0, 256); after the softmax has read it, O's value
// columns 256-511 go there and columns 0-255 go to [256, 512).  Each item
// writes its partial (o, row max, row sum), laid out so that the chunks of a
// (b, h) row are contiguous; a second kernel merges them.  Persistent grid,
// one CTA per SM: the whole chunks of all sequences are numbered first and
// the partial last chunks after them, and items are dealt round-robin, so
// with about one item per SM the short chunks are the ones that share an SM.
//
// Roles (320 threads): warps 0-7 softmax, two threads per head row (TMEM
// lane), warps 0-3 on the chunk's first 128 positions and warps 4-7 on the
// rest; warp 8 TMA producer, warp 9 MMA issuer.  A ring of three 48 KB
// stages carries, per item, the nine (Q box, K box) pairs of S; the same
// space then takes the eight value boxes (the first 512 columns of the same
// rows, now from L2) in pairs, two slots of two boxes 32 KB apart, so that
// each O step is one N = 128 product (sixteen N = 64 ones per box measured
// 2 us slower on the 24 x 128-head decode: small products pace O).
// Positions of a last chunk at or past lens[b] get zero weight, O's
// 16-position steps past the length are not issued, and the MMA warp zeroes
// the value rows past the length in the last step it issues, so whatever
// the cache holds there cannot reach the output.  The partial output is
// 256 KiB per item, about as long for an SM to write as the O products take
// to form, so warps 0-3 write it pair by pair as O completes, with plain
// stores (TMA stores would queue on the TMA unit ahead of the value loads).
#include "common.cuh"
#include "internal.h"

namespace cpattn {
namespace {

constexpr int kMdThreads = 320;
constexpr int kMdSoftmax = 256;            // softmax and epilogue threads (warps 0-7)
constexpr int kMdDk = 576, kMdDv = 512;
constexpr int kMdRows = 128;               // heads per MMA (rows past H are zero)
constexpr int kMdT = 256;                  // positions per chunk
constexpr int kMdKBoxes = kMdDk / 64;      // 9
constexpr int kMdVBoxes = kMdDv / 64;      // 8
constexpr int kMdNS = 3;                   // S ring stages
constexpr int kMdQBox = kMdRows * 128;   // 16 KB
constexpr int kMdKBox = kMdT * 128;      // 32 KB
constexpr int kMdStage = kMdQBox + kMdKBox;
// after S the ring's space takes the value boxes in pairs, two slots of two
// boxes 32 KB apart (one N = 128 operand of O), then the epilogue's staging
constexpr int kMdVPair = 2 * kMdKBox;               // 64 KB
constexpr int kMdNPairs = kMdVBoxes / 2;            // 4
constexpr int kMdOffE = 2 * kMdVPair;               // 16 KB of output staging
static_assert(kMdOffE + kMdQBox <= kMdNS * kMdStage && kMdNS == 3 && kMdKBoxes % kMdNS == 0,
              "slot A lies over S stages 0-1, slot B over 1-2, the staging inside stage 2");
constexpr int kMdOffP = kMdNS * kMdStage;          // P: 4 boxes of 64 positions x 128 rows
constexpr int kMdPBytes = 4 * kMdRows * 128;       // 64 KB
constexpr int kMdOffBar = kMdOffP + kMdPBytes;
constexpr int kMdOffMisc = kMdOffBar + 256;
constexpr int kMdOffRed = kMdOffMisc + 64;                      // row max and row sum of each half: [2][2][128] fp32
constexpr int kMdMaxB = 1024;
constexpr int kMdOffLens = kMdOffRed + 4 * kMdRows * 4;
constexpr int kMdOffPre = kMdOffLens + kMdMaxB * 4;            // whole chunks before each sequence
constexpr int kMdOffPre2 = kMdOffPre + (kMdMaxB + 1) * 4;       // partial chunks before each sequence
constexpr int kMdSmem = kMdOffPre2 + (kMdMaxB + 1) * 4 + 1024;
static_assert(kMdSmem <= 232448, "shared memory budget");
static_assert(kMdStage % 1024 == 0 && kMdOffP % 1024 == 0, "swizzled tiles need 1024-byte alignment");

struct MdBars {
  uint64_t full[kMdNS], empty[kMdNS];  // S ring
  uint64_t vfull[2], vempty[2];        // value pair slots
  uint64_t s_full, p_full, o_free, e_free;
  uint64_t o_pair[kMdNPairs];          // O's value pair p complete
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
    mbar_init(&bar.p_full, kMdSoftmax);
    mbar_init(&bar.o_free, kMdSoftmax);
    mbar_init(&bar.e_free, 1);
    for (int i = 0; i < 2; ++i) { mbar_init(&bar.vfull[i], 1); mbar_init(&bar.vempty[i], 1); }
    for (int i = 0; i < kMdNPairs; ++i) mbar_init(&bar.o_pair[i], 1);
    mbar_init(&bar.done, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 9) { tmem_alloc(tmem_slot, 512); tmem_relinquish(); }
  if (warp == 8 && lane == 0) { prefetch_tmap(&a.tq); prefetch_tmap(&a.tk); }
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

  if (warp == 8) {
    // ------------------------------------------------------------ TMA producer
    // item k: key box c (with its query box) in stage c % 3, that stage's
    // fill 3k + c / 3; then value pair p (boxes 2p, 2p + 1) in slot p & 1,
    // that slot's fill 2k + p / 2.  A region is filled again only once
    // everything that read it has released it: the first S stages of an
    // item wait for the previous item's value pairs (and the last one for
    // its output staging), the first pairs for the S stages under them.
    if (lane == 0) {
      bool ok = true;
      int sfill[kMdNS] = {0, 0, 0}, vfill[2] = {0, 0};
      for (int k = 0; k < n_items && ok; ++k) {
        const MdItem it = md_item(cta + k * ncta, pre, pre2, lens_s, a.B);
        for (int c = 0; c < kMdKBoxes; ++c) {
          const int st = c % kMdNS, f = (kMdKBoxes / kMdNS) * k + c / kMdNS;
          ok = mbar_wait(&bar.empty[st], (f & 1) ^ 1, ab);
          if (ok && k > 0 && c < kMdNS) {
            if (st <= 1) ok = mbar_wait(&bar.vempty[0], 1, ab);  // slot A's second fill of item k - 1 released
            if (ok && st >= 1) ok = mbar_wait(&bar.vempty[1], 1, ab);
            if (ok && st == 2) ok = mbar_wait(&bar.e_free, (k - 1) & 1, ab);
          }
          if (!ok) break;
          unsigned char* sb = smem + st * kMdStage;
          mbar_expect_tx(&bar.full[st], kMdStage);
          tma_load_3d(sb, &a.tq, &bar.full[st], c * 64, 0, it.b);
          tma_load_3d(sb + kMdQBox, &a.tk, &bar.full[st], c * 64, it.chunk * kMdT, it.b);
          ++sfill[st];
        }
        for (int p = 0; p < kMdNPairs && ok; ++p) {
          const int sl = p & 1;
          if (p < 2) {  // the S stages under the slot (0-1 for A, 1-2 for B) read out: their fill 3k + 2
            const uint32_t par = ((kMdKBoxes / kMdNS) * k + kMdKBoxes / kMdNS - 1) & 1;
            ok = mbar_wait(&bar.empty[sl], par, ab) && mbar_wait(&bar.empty[sl + 1], par, ab);
          } else {  // the slot's first pair of this item read out
            ok = mbar_wait(&bar.vempty[sl], 0, ab);
          }
          if (!ok) break;
          unsigned char* vb = smem + sl * kMdVPair;
          mbar_expect_tx(&bar.vfull[sl], kMdVPair);
          tma_load_3d(vb, &a.tk, &bar.vfull[sl], (2 * p) * 64, it.chunk * kMdT, it.b);
          tma_load_3d(vb + kMdKBox, &a.tk, &bar.vfull[sl], (2 * p + 1) * 64, it.chunk * kMdT, it.b);
          ++vfill[sl];
        }
      }
      if (!ok) {  // let the copies already issued land (each wait bounded on its own)
        for (int st = 0; st < kMdNS; ++st)
          if (sfill[st] > 0) {
            volatile int own = 0;
            mbar_wait(&bar.full[st], (sfill[st] - 1) & 1, Abort{&own, a.err});
          }
        for (int sl = 0; sl < 2; ++sl)
          if (vfill[sl] > 0) {
            volatile int own = 0;
            mbar_wait(&bar.vfull[sl], (vfill[sl] - 1) & 1, Abort{&own, a.err});
          }
      }
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    // lane 0 issues; the whole warp waits for each stage and slot in turn
    // (never more than one phase behind its barrier: a region is refilled
    // only after this warp's MMAs on it) and, in a partial chunk, zeroes the
    // value rows from the length up to the end of its last 16-position step,
    // the only rows past the length that O reads (its steps past that are
    // not issued): they come from a cache that may hold anything there
    constexpr uint32_t IDESC_S = idesc_bf16(kMdRows, kMdT, 0, 0);  // Q (K-major) x K (K-major)
    constexpr uint32_t IDESC_O = idesc_bf16(kMdRows, 128, 0, 1);   // P (K-major) x value pair (MN-major)
    const uint32_t s0 = smem_u32(smem);
    const uint64_t pdesc = sdesc_sw128(s0 + kMdOffP, 16, 1024);
    bool ok = true;
    for (int k = 0; k < n_items && ok; ++k) {
      const MdItem it = md_item(cta + k * ncta, pre, pre2, lens_s, a.B);
      const int nvalid = min(kMdT, it.len - it.chunk * kMdT);
      const int nk = (nvalid + 15) >> 4;  // 16-position steps of O that hold a valid position
      if (k > 0 && !(ok = __all_sync(0xffffffffu, mbar_wait(&bar.o_free, (k - 1) & 1, ab)))) break;  // the last O read out
      for (int c = 0; c < kMdKBoxes; ++c) {
        const int st = c % kMdNS, f = (kMdKBoxes / kMdNS) * k + c / kMdNS;
        if (!(ok = __all_sync(0xffffffffu, mbar_wait(&bar.full[st], f & 1, ab)))) break;
        if (lane == 0) {
          tc_fence_after();
          const uint64_t qd = sdesc_sw128(s0 + st * kMdStage, 16, 1024);
          const uint64_t kd = sdesc_sw128(s0 + st * kMdStage + kMdQBox, 16, 1024);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_ss(tmem, qd + ((kk * 32) >> 4), kd + ((kk * 32) >> 4), IDESC_S, (c > 0 || kk > 0) ? 1u : 0u);
          mma_commit(&bar.empty[st]);
        }
        __syncwarp();
      }
      if (!ok) break;
      if (lane == 0) mma_commit(&bar.s_full);
      // P written, S read: its columns take O
      if (!(ok = __all_sync(0xffffffffu, mbar_wait(&bar.p_full, k & 1, ab)))) break;
      for (int p = 0; p < kMdNPairs; ++p) {
        const int sl = p & 1;
        if (!(ok = __all_sync(0xffffffffu, mbar_wait(&bar.vfull[sl], (2 * k + (p >> 1)) & 1, ab)))) break;
        unsigned char* vb = smem + sl * kMdVPair;
        if (nvalid < 16 * nk) {
          for (int x = lane; x < (16 * nk - nvalid) * 16; x += 32) {  // 16-byte chunks, 8 per row in each box
            const int row = nvalid + (x >> 4), q = x & 15;
            *reinterpret_cast<uint4*>(vb + (q >> 3) * kMdKBox + row * 128 + (q & 7) * 16) = make_uint4(0, 0, 0, 0);
          }
          fence_proxy_async_smem();
          __syncwarp();
        }
        if (lane == 0) {
          tc_fence_after();
          // the pair's two 64-column boxes are the operand's MN blocks, 32 KB apart
          const uint64_t vd = sdesc_sw128(s0 + sl * kMdVPair, kMdKBox, 1024);
          for (int kk = 0; kk < nk; ++kk)
            mma_ss(tmem + (p < 2 ? 256 + 128 * p : 128 * (p - 2)),
                   pdesc + ((((kk >> 2) * (kMdRows * 128)) + (kk & 3) * 32) >> 4), vd + ((kk * 16 * 128) >> 4), IDESC_O,
                   kk > 0 ? 1u : 0u);
          mma_commit(&bar.vempty[sl]);
          mma_commit(&bar.o_pair[p]);
        }
        __syncwarp();
      }
    }
    if (lane == 0) mma_drain(&bar.done, a.err);
  } else if (warp < 8) {
    // ------------------------------------------------------------ softmax and epilogue
    // thread (r, hf): head row r = TMEM lane and half hf of the chunk's
    // positions in the softmax; then warps 0-3 write the partial output box
    // by box as O completes.  A failed wait runs on (every wait is bounded
    // and the barrier counts still complete)
    const int r = (warp & 3) * 32 + lane, hf = warp >> 2;
    const uint32_t lane_base = uint32_t((warp & 3) * 32) << 16;
    float* red = reinterpret_cast<float*>(smem + kMdOffRed);  // [0, 256): row max by half, [256, 512): row sum
    const float sl2 = a.scale_log2;
    for (int k = 0; k < n_items; ++k) {
      const MdItem it = md_item(cta + k * ncta, pre, pre2, lens_s, a.B);
      const int nvalid = min(kMdT, it.len - it.chunk * kMdT);  // positions of the chunk inside the cache
      mbar_wait(&bar.s_full, k & 1, ab);
      tc_fence_after();
      float m = -INFINITY;
#pragma unroll 1
      for (int c = 4 * hf; c < 4 * hf + 4; ++c) {
        uint32_t sv[32];
        tmem_ld32(tmem + lane_base + 32 * c, sv);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 32; ++j)
          if (32 * c + j < nvalid) m = fmaxf(m, __uint_as_float(sv[j]));
      }
      red[hf * kMdRows + r] = m;
      named_bar(3, kMdSoftmax);
      m = fmaxf(red[r], red[kMdRows + r]);  // finite: every item holds position 0 of its chunk
      const float m2 = m * sl2;
      float l = 0.f;
#pragma unroll 1
      for (int c = 4 * hf; c < 4 * hf + 4; ++c) {
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
      red[2 * kMdRows + hf * kMdRows + r] = l;
      tc_fence_before();
      fence_proxy_async_smem();
      mbar_arrive(&bar.p_full);
      if (hf == 0) {
        // epilogue, overlapping O: value pair p (columns 128p..128p+127) is
        // in TMEM [256 + 128p, ...) for p < 2 and [128(p-2), ...) after; it
        // goes out as four groups of 32 columns x 128 head rows, each staged
        // in shared memory (128-byte swizzle) and read back so that each warp
        // store writes four whole 128-byte lines of four heads' rows.  Plain
        // stores, not TMA: the TMA unit stays free for the value pairs that
        // O still waits for.  (Splitting this over two warp groups that pass
        // 16-column groups through two buffers measured 3% slower.)
        const size_t obase = ((size_t)it.b * a.H) * a.nch + it.chunk;  // partial row of (b, head 0, chunk)
        unsigned char* buf = smem + kMdOffE;
        const int q = r & 7;  // 16-byte piece of a head's 128-byte row, in the read-back
#pragma unroll 1
        for (int c = 0; c < kMdDv / 32; ++c) {
          if ((c & 3) == 0) {
            mbar_wait(&bar.o_pair[c >> 2], k & 1, ab);
            tc_fence_after();
          }
          uint32_t ov[32];
          tmem_ld32(tmem + lane_base + (c < 8 ? 256 + 32 * c : 32 * (c - 8)), ov);
          tmem_ld_wait();
          if (c > 0) named_bar(1, kMdRows);  // the previous group has been read back
          unsigned char* rp = buf + r * 128;
#pragma unroll
          for (int ch = 0; ch < 8; ++ch)
            *reinterpret_cast<uint4*>(rp + ((ch ^ (r & 7)) << 4)) =
                make_uint4(ov[4 * ch], ov[4 * ch + 1], ov[4 * ch + 2], ov[4 * ch + 3]);
          named_bar(1, kMdRows);
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const int head = (r >> 3) + 16 * j;
            if (head < a.H)
              *reinterpret_cast<uint4*>(a.part_o + (obase + (size_t)head * a.nch) * kMdDv + 32 * c + 4 * q) =
                  *reinterpret_cast<const uint4*>(buf + head * 128 + ((q ^ (head & 7)) << 4));
          }
        }
      }
      named_bar(3, kMdSoftmax);  // both halves' row sums are in; every O box has been read
      const size_t mrow = ((size_t)it.b * a.H + r) * a.nchp + it.chunk;
      if (hf == 0 && r < a.H) {
        a.part_ml[2 * mrow] = m2;
        a.part_ml[2 * mrow + 1] = red[2 * kMdRows + r] + red[3 * kMdRows + r];
      }
      tc_fence_before();
      mbar_arrive(&bar.o_free);
      if (tid == 0) mbar_arrive(&bar.e_free);  // the staging has been read back: the next item may load over it
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// merge of the chunks of each (b, h) row: one CTA of 128 threads per row,
// four value columns per thread, merged online.  The row's partials are
// contiguous ([b][h][chunk]); each thread copies its 16 bytes of eight
// chunks at a time into shared memory with cp.async (so no register holds a
// load in flight, and 16 KB of shared memory per CTA, not the register file,
// bounds how many rows are in flight on an SM) and reads them back.
// Launched as a programmatic dependent, so the partials are read only after
// the attention grid has completed.  (Loads into registers held 1520 rows in
// flight and took two waves over the 3072 rows of the 24 x 128-head decode;
// fetching each row's partials with bulk copies, twelve rows ahead on a
// persistent grid, measured three times slower: about 14 GB/s per SM.)
constexpr int kMgChunks = 8;
constexpr int kMgSmem = kMgChunks * kMdDv * 4;  // 16 KB
__device__ __forceinline__ void mg_cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__global__ void __launch_bounds__(128) mla_decode_merge_kernel(const __grid_constant__ MlaDecodeArgs a) {
  extern __shared__ float4 mg_x[];  // [chunk][thread]
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int row = blockIdx.x, b = row / a.H;
  int len = a.lens[b];
  len = len < 0 ? 0 : (len > a.Smax ? a.Smax : len);
  const int nch = (len + kMdT - 1) / kMdT;
  __nv_bfloat16* o = static_cast<__nv_bfloat16*>(a.out) + (size_t)row * kMdDv + 4 * threadIdx.x;
  if (nch == 0) {  // empty cache: zeros
    *reinterpret_cast<uint2*>(o) = make_uint2(0u, 0u);
    return;
  }
  const float4* po = reinterpret_cast<const float4*>(a.part_o + (size_t)row * a.nch * kMdDv) + threadIdx.x;
  const float2* pml = reinterpret_cast<const float2*>(a.part_ml + (size_t)row * a.nchp * 2);
  float M = -INFINITY, L = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int c0 = 0; c0 < nch; c0 += kMgChunks) {
    const int nc = min(kMgChunks, nch - c0);
    for (int j = 0; j < nc; ++j) mg_cp_async16(&mg_x[j * 128 + threadIdx.x], po + (size_t)(c0 + j) * (kMdDv / 4));
    asm volatile("cp.async.commit_group;" ::: "memory");
    float2 ml[kMgChunks];
#pragma unroll
    for (int j = 0; j < kMgChunks; ++j) ml[j] = __ldcg(pml + min(c0 + j, nch - 1));  // past the last chunk: weight 0 below
    asm volatile("cp.async.wait_all;" ::: "memory");  // this thread's own copies (it reads only those)
    float mn = M;
#pragma unroll
    for (int j = 0; j < kMgChunks; ++j)
      if (j < nc) mn = fmaxf(mn, ml[j].x);  // finite: chunk c0 is in
    const float f = fast_exp2(M - mn);
    L *= f;
    acc.x *= f;
    acc.y *= f;
    acc.z *= f;
    acc.w *= f;
#pragma unroll
    for (int j = 0; j < kMgChunks; ++j)
      if (j < nc) {
        const float w = fast_exp2(ml[j].x - mn);
        const float4 x = mg_x[j * 128 + threadIdx.x];
        L = fmaf(ml[j].y, w, L);
        acc.x = fmaf(x.x, w, acc.x);
        acc.y = fmaf(x.y, w, acc.y);
        acc.z = fmaf(x.z, w, acc.z);
        acc.w = fmaf(x.w, w, acc.w);
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
  if (encode_tmap(&a.tq, a.q, 3, qd, qs, qb, 2) || encode_tmap(&a.tk, a.ckv, 3, kd, ks, kb, 2))
    return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(mla_decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kMdSmem);
  if (e != cudaSuccess) return e;
  mla_decode_kernel<<<num_sms, kMdThreads, kMdSmem, st>>>(a);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.B * a.H);
  cfg.blockDim = dim3(128);
  cfg.dynamicSmemBytes = kMgSmem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, mla_decode_merge_kernel, a);
}

}  // namespace cpattn
