// Shared device helpers for the cpattn kernels (sm_103a only).
//
//  * Load-balance position map: the reorder of "Add context parallelism"
//    (MaxText pull request 1445), Description -- 2*cp chunks of c tokens,
//    shard s holds chunk s then chunk 2cp-1-s, so memory slot j holds the
//    token at original position pos(j).  Closed form, usable on host and
//    device, plus tile range queries used by the work scheduler.
//  * Hand-written PTX wrappers: mbarrier (bounded waits that raise an error
//    flag instead of hanging), TMA tiled loads, tcgen05 MMA / TMEM access.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>
#include <cuda.h>
#include <cuda_bf16.h>

#ifndef CPATTN_HD
#define CPATTN_HD __host__ __device__ __forceinline__
#endif

namespace cpattn {

// device error codes written into the per-device error word
enum : int {
  DEV_OK = 0,
  DEV_TIMEOUT = 1,      // a bounded mbarrier wait ran out
  DEV_LENS_CLAMPED = 2, // gqa_decode saw lens[b] outside [0, Smax]
  DEV_SMEM_ALIGN = 3,   // dynamic shared memory not 1024-byte aligned (kernel did nothing)
};

constexpr int kMaxPieces = 64;

// ---------------------------------------------------------------------------
// position map
// ---------------------------------------------------------------------------
struct PosMap {
  int S;   // sequence length
  int cp;  // number of shards
  int lb;  // 0: natural order; 1: tensors in load-balanced slot order; 2: tensors in
           // natural order, load-balanced schedule (slot j lives at memory row pos(j))
  int c;   // chunk length S/(2cp) (only meaningful when lb)

  CPATTN_HD static PosMap make(int S_, int cp_, int load_balance) {
    PosMap m;
    m.S = S_;
    m.cp = cp_;
    m.lb = (load_balance && cp_ > 1) ? (load_balance == 2 ? 2 : 1) : 0;
    m.c = m.lb ? S_ / (2 * cp_) : S_;
    return m;
  }
  // memory row of slot j (a whole tile of slots is contiguous in memory when
  // the chunk length is a multiple of the tile)
  CPATTN_HD int row(int slot) const { return lb == 2 ? pos(slot) : slot; }
  // original chunk held by memory chunk k
  CPATTN_HD int chunk_of(int k) const {
    int s = k >> 1;
    return (k & 1) ? (2 * cp - 1 - s) : s;
  }
  // memory chunk holding original chunk ch
  CPATTN_HD int mem_chunk_of(int ch) const {
    return ch < cp ? 2 * ch : 2 * (2 * cp - 1 - ch) + 1;
  }
  CPATTN_HD int pos(int slot) const {
    if (!lb) return slot;
    int k = slot / c;
    int t = slot - k * c;
    return chunk_of(k) * c + t;
  }
  CPATTN_HD int slot(int p) const {
    if (!lb) return p;
    int ch = p / c;
    int t = p - ch * c;
    return mem_chunk_of(ch) * c + t;
  }
  // min and max original position over slots [a, b) (b clipped to S)
  CPATTN_HD void range(int a, int b, int& mn, int& mx) const {
    if (b > S) b = S;
    if (!lb) { mn = a; mx = b - 1; return; }
    mn = 0x7fffffff;
    mx = -1;
    while (a < b) {
      int k = a / c;
      int e = (k + 1) * c;
      if (e > b) e = b;
      int base = chunk_of(k) * c - k * c;
      int p0 = base + a, p1 = base + e - 1;
      mn = p0 < mn ? p0 : mn;
      mx = p1 > mx ? p1 : mx;
      a = e;
    }
  }
};

// Tile list walkers.  Tiles have T slots; tile t covers slots [tT, tT+T).
//  next_kv_tile: next tile (> cur) whose min position is <= bound, i.e. a
//    key tile that query rows with position <= bound may see.
//  next_q_tile: next tile (> cur) whose max position is >= bound, i.e. a
//    query tile with at least one row that sees a key at position bound.
// When every chunk is a whole number of tiles the walk jumps over chunks
// that cannot qualify, so a walk costs O(chunks + visited tiles).
CPATTN_HD int next_kv_tile(const PosMap& m, int T, int cur, int bound) {
  const int nt = (m.S + T - 1) / T;
  int t = cur + 1;
  if (!m.lb) return (t * T <= bound && t < nt) ? t : -1;
  if (m.c % T == 0) {
    const int tpc = m.c / T;
    while (t < nt) {
      int k = t / tpc;
      int p0 = m.chunk_of(k) * m.c + (t - k * tpc) * T;
      if (p0 <= bound) return t;
      t = (k + 1) * tpc;  // rest of this chunk starts even later
    }
    return -1;
  }
  for (; t < nt; ++t) {
    int mn, mx;
    m.range(t * T, t * T + T, mn, mx);
    if (mn <= bound) return t;
  }
  return -1;
}

// The key tiles of next_kv_tile, walked with their position range [kmin,
// kmax] and without an integer division per tile where every chunk is a
// whole number of tiles (or there is no reorder): the walk keeps the tile's
// chunk, its offset in the chunk and its first position.  Otherwise each
// step falls back to next_kv_tile and PosMap::range.
struct KvWalk {
  int t, kmin, kmax;        // current tile (-1 after the last) and its positions
  int nt, T, bound, tpc, k, off;
  bool inc;

  CPATTN_HD void start(const PosMap& m, int T_, int bound_) {
    T = T_;
    bound = bound_;
    nt = (m.S + T - 1) / T;
    inc = !m.lb || m.c % T == 0;
    if (!inc) {
      t = next_kv_tile(m, T, -1, bound);
      fill(m);
      return;
    }
    tpc = m.lb ? m.c / T : nt;
    t = 0;
    k = 0;
    off = 0;
    kmin = 0;  // chunk_of(0) = 0
    settle(m);
  }
  CPATTN_HD void next(const PosMap& m) {
    if (!inc) {
      t = next_kv_tile(m, T, t, bound);
      fill(m);
      return;
    }
    ++t;
    kmin += T;
    if (++off == tpc) {
      ++k;
      off = 0;
      if (m.lb) kmin = m.chunk_of(k) * m.c;
    }
    settle(m);
  }

 private:
  // skip the rest of every chunk whose next tile starts past the bound
  CPATTN_HD void settle(const PosMap& m) {
    if (!m.lb) {
      if (t >= nt || kmin > bound) { t = -1; return; }
      kmax = kmin + T - 1 < m.S - 1 ? kmin + T - 1 : m.S - 1;
      return;
    }
    while (t < nt && kmin > bound) {
      ++k;
      off = 0;
      t = k * tpc;
      kmin = m.chunk_of(k) * m.c;
    }
    if (t >= nt) { t = -1; return; }
    kmax = kmin + T - 1;
  }
  CPATTN_HD void fill(const PosMap& m) {
    if (t >= 0) m.range(t * T, t * T + T, kmin, kmax);
  }
};

CPATTN_HD int next_q_tile(const PosMap& m, int T, int cur, int bound) {
  const int nt = (m.S + T - 1) / T;
  int t = cur + 1;
  if (!m.lb) {
    int first = bound / T;
    if (t < first) t = first;
    return t < nt ? t : -1;
  }
  if (m.c % T == 0) {
    const int tpc = m.c / T;
    while (t < nt) {
      int k = t / tpc;
      int pend = m.chunk_of(k) * m.c + (t - k * tpc) * T + T - 1;
      if (pend >= bound) return t;
      int chunk_last = m.chunk_of(k) * m.c + m.c - 1;
      if (chunk_last < bound) { t = (k + 1) * tpc; continue; }
      ++t;
    }
    return -1;
  }
  for (; t < nt; ++t) {
    int mn, mx;
    m.range(t * T, t * T + T, mn, mx);
    if (mx >= bound) return t;
  }
  return -1;
}

#ifdef __CUDACC__
// ---------------------------------------------------------------------------
// PTX wrappers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try(uint32_t addr, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(addr), "r"(parity)
      : "memory");
  return ok != 0;
}

constexpr long long kWaitLimitCycles = 4000000000LL;  // about two seconds

// Abort state shared by all roles of a CTA.  A wait that runs out of time
// (limit SM clock cycles) records DEV_TIMEOUT in the global error word and
// raises the CTA's abort flag; every other wait then gives up promptly, the
// roles leave their loops and the CTA frees its TMEM and exits.
struct Abort {
  volatile int* flag;  // shared memory
  int* err;            // global error word
  long long limit = kWaitLimitCycles;
};

__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, const Abort& ab) {
  const uint32_t a = smem_u32(bar);
  if (mbar_try(a, parity)) return true;
  const long long t0 = clock64();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try(a, parity)) return true;
    if ((it & 63) == 0) {
      if (*ab.flag) return false;
      if (clock64() - t0 > ab.limit) {
        *ab.flag = 1;
        atomicExch(ab.err, DEV_TIMEOUT);
        __threadfence_block();
        return false;
      }
    }
  }
}

// TMA: 4-D tiled load global -> shared, completion counted on an mbarrier
__device__ __forceinline__ void tma_load_4d(void* dst, const CUtensorMap* map, uint64_t* bar, int c0,
                                            int c1, int c2, int c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
      : "memory");
}
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, uint64_t* bar, int c0, int c1,
                                            int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}
// make this thread's generic-proxy shared-memory writes visible to the async proxy (TMA, tensor core)
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// TMA: fetch a tile of a 4-D tensor into L2 ahead of its load (no shared
// memory, no barrier; a hint the hardware may drop)
__device__ __forceinline__ void tma_prefetch_l2_4d(const CUtensorMap* map, int c0, int c1, int c2, int c3) {
  asm volatile("cp.async.bulk.prefetch.tensor.4d.L2.global.tile [%0, {%1, %2, %3, %4}];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(c0), "r"(c1), "r"(c2), "r"(c3)
               : "memory");
}
// plain bulk copy global -> shared (16-byte aligned, size multiple of 16)
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ---- tcgen05 -------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// D[tmem] (+)= A[smem] * B[smem]
__device__ __forceinline__ void mma_ss(uint32_t d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                       uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(acc)
      : "memory");
}
// D[tmem] (+)= A[tmem] * B[smem]
__device__ __forceinline__ void mma_ts(uint32_t d, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                       uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(acc)
      : "memory");
}
// arrive on an mbarrier once every tcgen05 op issued so far by this thread completes
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}

// Commit, then wait until every tcgen05 operation this thread issued has
// completed, before the CTA releases its TMEM.  Bounded, but it does not give
// up on the CTA's abort flag: after an abort the MMAs already issued still
// complete (they wait on nothing), and TMEM must not be freed under them.
__device__ __forceinline__ void mma_drain(uint64_t* done, int* err, long long limit = kWaitLimitCycles) {
  mma_commit(done);
  volatile int own = 0;
  mbar_wait(done, 0, Abort{&own, err, limit});
}

// instruction descriptor, kind::f16 with bf16 A/B and fp32 accumulation
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, int a_mn_major, int b_mn_major) {
  return (1u << 4)                        // D format f32
         | (1u << 7)                      // A format bf16
         | (1u << 10)                     // B format bf16
         | (uint32_t(a_mn_major) << 15)   // A major-ness
         | (uint32_t(b_mn_major) << 16)   // B major-ness
         | (uint32_t(N >> 3) << 17)       // N / 8
         | (uint32_t(M >> 4) << 24);      // M / 16
}

// shared-memory matrix descriptor, 128-byte swizzle
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= uint64_t((saddr & 0x3FFFF) >> 4);
  d |= uint64_t((lbo >> 4) & 0x3FFF) << 16;
  d |= uint64_t((sbo >> 4) & 0x3FFF) << 32;
  d |= uint64_t(1) << 46;  // descriptor version for tcgen05
  d |= uint64_t(2) << 61;  // 128-byte swizzle
  return d;
}

// TMEM loads/stores: 32 lanes x 32 bit, 32 consecutive columns per thread
#define CPATTN_R32(r)                                                                        \
  "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),        \
      "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), \
      "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),          \
      "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),          \
      "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
#define CPATTN_W32(r)                                                                           \
  "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),       \
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),         \
      "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),       \
      "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),       \
      "r"(r[29]), "r"(r[30]), "r"(r[31])

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, "
      "%12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, "
      "%30, %31}, [%32];"
      : CPATTN_R32(r)
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, "
      "%29, %30, %31, %32};" ::"r"(taddr),
      CPATTN_W32(r)
      : "memory");
}

#define CPATTN_R16(r)                                                                              \
  "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), \
      "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),     \
      "=r"(r[15])
#define CPATTN_W16(r)                                                                                 \
  "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), \
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, "
      "%12, %13, %14, %15}, [%16];"
      : CPATTN_R16(r)
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      CPATTN_W16(r)
      : "memory");
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// r-th unit of CTA `cta`: the host deals the work list out CTA by CTA (CTA c
// runs units [off[c], off[c+1]) in that order); -1 past the CTA's last unit
__device__ __forceinline__ int unit_index(const int* __restrict__ off, int r, int cta) {
  const int ui = off[cta] + r;
  return ui < off[cta + 1] ? ui : -1;
}

// Two element-wise groups each own HC consecutive TMEM columns of a row; a
// group packs the bf16 pairs of column c into its own range, so the packed
// column of c is (c / HC) * HC + (c % HC) / 2.  TS MMAs read 16 columns (8
// packed) per k-step, never straddling two groups.
template <int HC>
__host__ __device__ constexpr int packed_col(int c) { return (c / HC) * HC + (c % HC) / 2; }

// TMA reduce-add of a tile from shared memory into global memory (element
// type of the tensor map), tracked by the issuing thread's bulk async-group
__device__ __forceinline__ void tma_reduce_add_4d(const void* src, const CUtensorMap* map, int c0, int c1, int c2,
                                                  int c3) {
  asm volatile(
      "cp.reduce.async.bulk.tensor.4d.global.shared::cta.add.tile.bulk_group [%0, {%2, %3, %4, %5}], [%1];" ::"l"(
          reinterpret_cast<uint64_t>(map)),
      "r"(smem_u32(src)), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
      : "memory");
}
__device__ __forceinline__ void bulk_commit_group() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// this thread's bulk groups have finished reading their shared-memory sources
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// ... and their writes are complete
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// named barrier among `count` threads
__device__ __forceinline__ void named_bar(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// two fp32 -> packed bf16x2 (lo in the low half), round to nearest even
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ float bf16lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ int elect_one_lane() { return (threadIdx.x & 31) == 0; }

// packed fp32 pairs (Blackwell f32x2 arithmetic: one instruction, two lanes of math)
__device__ __forceinline__ uint64_t f2pack(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ uint64_t f2pack_u(uint32_t a, uint32_t b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "r"(a), "r"(b));
  return r;
}
__device__ __forceinline__ void f2unpack(uint64_t r, float& a, float& b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(r));
}
__device__ __forceinline__ uint64_t f2fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
__device__ __forceinline__ uint64_t f2add(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t f2mul(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// register re-balancing between warpgroups (all warps of a warpgroup execute it)
template <int N>
__device__ __forceinline__ void regs_inc() { asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N)); }
template <int N>
__device__ __forceinline__ void regs_dec() { asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N)); }
#endif  // __CUDACC__

}  // namespace cpattn
