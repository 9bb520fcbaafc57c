// Fused flash backward for equal query/key and value head dims (64 or 128).
//
// Same gradient as the two-kernel backward (the textbook gradient of
// out = softmax(scale q k^T + mask) v under the reordered causal mask), but
// in one pass: a CTA owns a 128-row key tile of one KV head and walks every
// (query head of the group, 128-row query tile) that sees it.  Per step, on
// tcgen05 with 128-wide N throughout:
//   S^T  = K Q^T            (TMEM, key lanes)  -> P^T  (bf16, in place)
//   dP^T = V dO^T           (TMEM, key lanes)  -> dS^T (bf16, in place) and
//                                                 dS    (bf16, shared memory)
//   dV  += P^T dO,  dK += dS^T Q               (TMEM accumulators)
//   dQ_step = dS K          (TMEM, query lanes, in dP's columns)
// and dQ_step is scaled and added into an fp32 dQ accumulator in global
// memory with TMA reduce-add (so S and dP are formed once, not twice as in
// the dQ kernel of the two-kernel path).  The accumulator is zeroed by the
// preprocess kernel and rounded to bf16 by a final pass.
//
// MMA order per step j:  dP_j, dV_j, S_{j+1}, dK_j, dQ_j; the element-wise
// warps run P_{j+1} while dK_j and dQ_j execute, then form dS_{j+1} while
// dV_{j+1} and S_{j+2} execute.  dQ_j is taken out of TMEM by a warpgroup of
// its own the moment it is complete, because dP_{j+1} needs its columns and
// the tensor core waits for them.  TMEM (512 columns): S/P 128, dP/dS/dQ
// 128, dV D, dK D.  Tensor-core MMAs from one thread execute in issue order,
// so an MMA may overwrite TMEM columns an earlier one reads.
//
// Shared memory (D = 128, 226 KiB): K and V tiles (resident per unit), two
// stages each of Q and dO with the per-row -lse*log2(e) and -D vectors, and
// one dS tile.  dQ_step (128 x D fp32) is staged for the reduce in the dS
// tile and, for D = 128, in the step's dO stage (both dead by then; the Q
// stage is not, since S_{j+1} reads the other one and Q_{j+2} must land in
// this one by the next step).  The dS tile's chunks are staged first and
// reduced as soon as they are (the next step's dS waits for that space, and
// that wait is on the MMA chain; timing trials showed reducing them first
// worth 2-5%, freeing the dO stage first instead cost 20-30%).
#include <cstdio>

#include "common.cuh"
#include "internal.h"

namespace cpattn {
namespace {

// warps 0-7 element-wise (two column halves), 8 TMA producer, 9 MMA issuer,
// 10 dQ reducer, 11 idle, 12-15 dQ read-out.  setmaxnreg moves registers from
// warpgroup 2 (producer, MMA, reducer) and warpgroup 3 (read-out) to the
// element-wise warpgroups.
constexpr int kThreadsF = 512;
constexpr int kRegsLaunchF = 128;  // 65536 / 512
constexpr int kRegsEw = 152;
constexpr int kRegsWg2 = 112;
constexpr int kRegsWg3 = 96;
static_assert(256 * kRegsEw + 128 * kRegsWg2 + 128 * kRegsWg3 <= kThreadsF * kRegsLaunchF, "register split");
// a warpgroup's share is set with setmaxnreg.inc when it grows from the launch
// count and .dec when it shrinks (either one in the other direction is invalid)
template <int N>
__device__ __forceinline__ void regs_to() {
  static_assert(N % 8 == 0 && N >= 24 && N <= 256, "setmaxnreg range");
  if constexpr (N > kRegsLaunchF) regs_inc<N>();
  else if constexpr (N < kRegsLaunchF) regs_dec<N>();
}
constexpr int kRows = 128;      // key rows per unit, query rows per step

template <int D>
struct FCfg {
  static constexpr int TILE = kRows * D * 2;  // D/64 boxes of 128 rows x 128 B
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = TILE;
  static constexpr int OFF_Q = 2 * TILE;   // stage s at OFF_Q + s*TILE
  static constexpr int OFF_DO = 4 * TILE;  // stage s at OFF_DO + s*TILE
  static constexpr int OFF_DS = 6 * TILE;  // dS as two query halves x 128 key rows x 128 B
  static constexpr int DS_BYTES = 2 * kRows * 128;
  static constexpr int OFF_VEC = OFF_DS + DS_BYTES;  // stage s: lse[128] then delta[128] (fp32)
  static constexpr int VEC_BYTES = 2 * kRows * 4;
  static constexpr int OFF_BAR = OFF_VEC + 2 * VEC_BYTES;
  static constexpr int OFF_MISC = OFF_BAR + 256;  // TMEM address, abort flag, StepInfo[2] at +32
  static constexpr int OFF_MROW = OFF_MISC + 64;  // memory row of each key row of the unit (-1 past S)
  static constexpr int SMEM = OFF_MROW + kRows * 4;
  static_assert(SMEM <= 232448, "shared memory budget");
  static_assert(TILE % 1024 == 0 && OFF_DS % 1024 == 0, "swizzled tiles need 1024-byte alignment");
  // TMEM columns
  static constexpr int T_S = 0;
  static constexpr int T_DP = 128;
  static constexpr int T_DV = 256;
  static constexpr int T_DK = 256 + D;
  static_assert(T_DK + D <= 512, "TMEM budget");
  static constexpr int NBOX = D / 32;  // fp32 dQ boxes of 32 columns x 128 rows (16 KiB)
};

// what the producer publishes with each Q stage: the step's query head and
// tile, and whether it is the last step of its unit (walking the steps costs
// a chain of integer divisions; only the producer, which runs ahead, pays it)
struct StepInfo {
  int hq, qt, last, qmin;  // qmin: first position of the query tile (decides the masked path)
};

struct FBars {
  uint64_t kv_full, kv_empty;
  uint64_t q_full[2], q_empty[2], do_full[2], do_empty[2];
  uint64_t s_full, p_full, dp_full, dst_full, dss_full, dq_full, dq_free, staged, staged_ds, ds_free;
  uint64_t acc_full, done;
};

// this thread's bulk async-groups, all but the newest N, have read their sources
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

// P for this thread's 64 query columns of one step: scores from TMEM (t_s),
// p = exp2(s * scale*log2e - lse*log2e), zeroed where the key's position is
// past the query's (MASKED steps only; positions walked slot by slot from
// slot0), kept in fp32 for dS and stored back to TMEM (t_pk) as packed bf16
template <bool MASKED, bool SHARD>
__device__ __forceinline__ void ew_p(uint32_t t_s, uint32_t t_pk, const float* lse_s, uint64_t sl2x2,
                                     float (&p)[64], int kpos, const PosMap& pm, int slot0, int lo, int hi) {
  int ck = 0, ct = 0, cbase = 0;  // memory chunk, offset in it, first position of the chunk
  if (MASKED && pm.lb) {
    ck = slot0 / pm.c;
    ct = slot0 - ck * pm.c;
    cbase = pm.chunk_of(ck) * pm.c;
  }
  auto next_qpos = [&](int slot) {
    int q = -1;
    if (slot < pm.S) {
      if (!pm.lb) {
        q = slot;
      } else {
        q = cbase + ct;
        if (++ct == pm.c) {
          ++ck;
          ct = 0;
          cbase = pm.chunk_of(ck) * pm.c;
        }
      }
    }
    return (!SHARD || (slot >= lo && slot < hi)) ? q : -1;  // rows outside [lo, hi) take no part
  };
  uint32_t sv[2][32];
  tmem_ld32(t_s, sv[0]);
  tmem_ld32(t_s + 32, sv[1]);
  tmem_ld_wait();
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const uint64_t* nl2 = reinterpret_cast<const uint64_t*>(lse_s + 32 * h);
    uint32_t pk[16];
#pragma unroll
    for (int c = 0; c < 32; c += 2) {
      float p0, p1;
      f2unpack(f2fma(f2pack_u(sv[h][c], sv[h][c + 1]), sl2x2, nl2[c >> 1]), p0, p1);
      p0 = fast_exp2(p0);
      p1 = fast_exp2(p1);
      if (MASKED) {
        const int q0 = next_qpos(slot0 + 32 * h + c);
        const int q1 = next_qpos(slot0 + 32 * h + c + 1);
        p0 = kpos <= q0 ? p0 : 0.f;
        p1 = kpos <= q1 ? p1 : 0.f;
      }
      p[32 * h + c] = p0;
      p[32 * h + c + 1] = p1;
      pk[c >> 1] = pack_bf16(p0, p1);
    }
    tmem_st16(t_pk + 16 * h, pk);
  }
}

// (query head, query tile) steps of a key-tile unit: the query tiles that
// see the key tile (and, per shard, hold a slot in [lo, hi)).
// Where every tile of slots is one tile of positions (no reorder, or chunks
// that are whole tiles, which natural-order tensors always have), the tiles
// are walked by DESCENDING position: from the last tile of the sequence down
// to the one holding the key tile's first position.  Every key tile of a head
// sees the top of the sequence, so the CTAs working on key tiles of the same
// head start on the same query tile and move through the same Q/dO tiles (and
// the same dQ accumulator rows) at about the same time: those tiles come from
// DRAM once and from L2 for the others.  Permuted and natural-order tensors
// go through the same steps in the same order.  The walk keeps the chunk and
// the offset in it of the current position tile, so a step costs no integer
// division (the producer computes it on the path that feeds the MMAs).
// Otherwise (chunks that are not whole tiles, or one shard's steps) the tiles
// are walked in slot order.
template <bool SHARD, bool NAT>
struct StepIter {
  int h_end, kmin, lo, hi;
  bool posw;              // walk by descending position
  int tpc, first, top;    // tiles per chunk; position tiles holding kmin and the sequence's end
  int hq, qt, pt, ch, off;  // current step: query head, slot tile, position tile, its chunk and offset

  __device__ __forceinline__ void init(const PosMap& pm, int h0, int h_end_, int kmin_, int lo_, int hi_) {
    h_end = h_end_;
    kmin = kmin_;
    lo = lo_;
    hi = hi_;
    hq = h0;
    posw = !SHARD && (NAT || pm.lb == 0 || pm.c % kRows == 0);
    tpc = pm.lb ? pm.c / kRows : 1;
    first = kmin / kRows;
    top = (pm.S + kRows - 1) / kRows - 1;
  }
  __device__ __forceinline__ void to_top(const PosMap& pm) {
    pt = top;
    if (pm.lb) {
      ch = 2 * pm.cp - 1;
      off = tpc - 1;
      qt = pm.mem_chunk_of(ch) * tpc + off;
    } else {
      qt = pt;
    }
  }
  __device__ __forceinline__ int slot_order_tile(const PosMap& pm, int cur) const {
    if (!SHARD) return next_q_tile(pm, kRows, cur, kmin);
    if (cur < 0) cur = lo / kRows - 1;  // no tile before the shard's first can qualify
    for (cur = next_q_tile(pm, kRows, cur, kmin); cur >= 0; cur = next_q_tile(pm, kRows, cur, kmin)) {
      if (cur * kRows >= hi) return -1;  // tiles come in increasing slot order
      if (cur * kRows + kRows > lo) return cur;
    }
    return -1;
  }
  // first step of the unit; false if no query tile sees the key tile
  __device__ __forceinline__ bool begin(const PosMap& pm) {
    if (posw) {  // the top tile sees every key
      to_top(pm);
      return true;
    }
    for (;; ) {
      qt = slot_order_tile(pm, -1);
      if (qt >= 0) return true;
      if (++hq >= h_end) return false;
    }
  }
  // advance to the next step; false after the unit's last one
  __device__ __forceinline__ bool next(const PosMap& pm) {
    if (posw) {
      if (pt > first) {
        --pt;
        if (pm.lb) {
          if (--off < 0) {
            --ch;
            off = tpc - 1;
          }
          qt = pm.mem_chunk_of(ch) * tpc + off;
        } else {
          qt = pt;
        }
        return true;
      }
      if (++hq >= h_end) return false;
      to_top(pm);
      return true;
    }
    qt = slot_order_tile(pm, qt);
    if (qt >= 0) return true;
    if (++hq >= h_end) return false;
    qt = slot_order_tile(pm, -1);
    return qt >= 0;
  }
  // first position of the current query tile (a position tile's own when
  // walking by position; otherwise from the slot range)
  __device__ __forceinline__ int qmin(const PosMap& pm) const {
    if (posw) return pt * kRows;
    int mn, mx;
    pm.range(qt * kRows, qt * kRows + kRows, mn, mx);
    return mn;
  }
  // memory row of the current query tile: natural-order tensors keep a
  // position tile at its position, the others a slot tile at its slot
  __device__ __forceinline__ int mem_row() const { return NAT ? pt * kRows : qt * kRows; }
};

// memory row of slot `slot`: natural-order tensors (NAT, load_balance 2) keep
// slot j at row pos(j); permuted or natural tensors without the reorder at row j
template <bool NAT>
__device__ __forceinline__ int mem_row(const PosMap& pm, int slot) { return NAT ? pm.pos(slot) : slot; }

// SHARD: only query slots [a.q_lo, a.q_hi) take part and dk/dv also go out
// as fp32 partials.  NAT: tensors in natural order (zero-copy load balance).
// Each is its own instantiation, so the plain backward keeps none of that
// bookkeeping in its code.
template <int D, bool SHARD, bool NAT>
__global__ void __launch_bounds__(kThreadsF, 1) attn_bwd_fused_kernel(const __grid_constant__ BwdArgs a) {
  using C = FCfg<D>;
  extern __shared__ __align__(1024) unsigned char smem[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // every offset below assumes a 1024-byte aligned base (no slack is left for
  // aligning by hand); a misaligned base is reported and the CTA does nothing
  if (smem_u32(smem) & 1023u) {
    if (tid == 0) atomicExch(a.err, DEV_SMEM_ALIGN);
    return;
  }
  FBars& bar = *reinterpret_cast<FBars*>(smem + C::OFF_BAR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 16);
  volatile StepInfo* info = reinterpret_cast<volatile StepInfo*>(smem + C::OFF_MISC + 32);
  const PosMap pm = PosMap::make(a.sh.S, a.sh.cp, a.sh.lb);
  const Abort ab{abort_flag, a.err};
  const int G = a.sh.Hq / a.sh.Hkv;
  const int cta = blockIdx.x;

  if (tid == 0) {
    mbar_init(&bar.kv_full, 1);
    mbar_init(&bar.kv_empty, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bar.q_full[i], 1);
      mbar_init(&bar.q_empty[i], 1);
      mbar_init(&bar.do_full[i], 1);
      mbar_init(&bar.do_empty[i], 1);
    }
    mbar_init(&bar.s_full, 1);
    mbar_init(&bar.p_full, 256);
    mbar_init(&bar.dp_full, 1);
    mbar_init(&bar.dst_full, 256);
    mbar_init(&bar.dss_full, 256);
    mbar_init(&bar.dq_full, 1);
    mbar_init(&bar.dq_free, 128);
    mbar_init(&bar.staged, 128);
    mbar_init(&bar.staged_ds, 128);
    mbar_init(&bar.ds_free, 1);
    mbar_init(&bar.acc_full, 1);
    mbar_init(&bar.done, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 9) { tmem_alloc(tmem_slot, 512); tmem_relinquish(); }
  if (warp == 8 && lane == 0) {
    prefetch_tmap(&a.tq); prefetch_tmap(&a.tk); prefetch_tmap(&a.tv); prefetch_tmap(&a.tdo); prefetch_tmap(&a.tdq);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  auto dq_readout = [&]() {
    // ------------------------------------------------------------ dQ read-out
    // dQ_j (query rows = TMEM lanes, D fp32 columns in dP's space): TMEM ->
    // registers -> shared memory for the reducer (the dS tile and, for
    // D = 128, the step's dO stage; boxes of 32 columns, 128-byte swizzle),
    // each 32-column chunk staged while the next load is in flight; the
    // columns are released as soon as the last load is done.  Both spaces are
    // dead once dQ_j is complete: dS_j and dO_j were last read by MMAs that
    // precede it.  The tile goes out unscaled (the final rounding pass applies
    // the softmax scale).
    const int qd = warp & 3;
    const int row = (qd << 5) + lane;  // query row of the tile == TMEM lane
    const uint32_t t_dq = tmem + (uint32_t(qd * 32) << 16) + C::T_DP;
    auto stage = [&](int gsr, int c, const uint32_t (&o)[32]) {
      unsigned char* bb = c < 2 ? smem + C::OFF_DS + c * (kRows * 128)
                                : smem + C::OFF_DO + (gsr & 1) * C::TILE + (c - 2) * (kRows * 128);
      unsigned char* rp = bb + row * 128;
#pragma unroll
      for (int ch = 0; ch < 8; ++ch)
        *reinterpret_cast<uint4*>(rp + ((ch ^ (row & 7)) << 4)) =
            make_uint4(o[4 * ch + 0], o[4 * ch + 1], o[4 * ch + 2], o[4 * ch + 3]);
    };
    int gs = 0;
    for (int r = 0;; ++r) {
      const int ui = unit_index(a.cta_off, r, cta);
      if (ui < 0) break;
      const BwdUnit u = a.units[ui];
      int kmin, kmax;
      pm.range(u.t * kRows, u.t * kRows + kRows, kmin, kmax);
      StepIter<SHARD, NAT> it;
      it.init(pm, u.h * G, u.h * G + G, kmin, a.q_lo, a.q_hi);
      if (!it.begin(pm)) continue;
      do {
        mbar_wait(&bar.dq_full, gs & 1, ab);  // runs on after an abort: the staging is garbage, the waits bounded
        tc_fence_after();
        uint32_t o[2][32];
        tmem_ld32(t_dq, o[0]);
        tmem_ld32(t_dq + 32, o[1]);
        tmem_ld_wait();
        if (C::NBOX > 2) {
          stage(gs, 0, o[0]);
          tmem_ld32(t_dq + 64, o[0]);
          stage(gs, 1, o[1]);
          tmem_ld32(t_dq + 96, o[1]);
          // the dS tile's chunks are staged: the reducer may add them (and
          // free the tile for the next dS) while the rest is read out
          fence_proxy_async_smem();
          mbar_arrive(&bar.staged_ds);
          tmem_ld_wait();
        }
        tc_fence_before();
        mbar_arrive(&bar.dq_free);
        stage(gs, C::NBOX - 2, o[0]);
        stage(gs, C::NBOX - 1, o[1]);
        fence_proxy_async_smem();
        mbar_arrive(&bar.staged);
        ++gs;
      } while (it.next(pm));
    }
  };

  // each role's code sits under its own setmaxnreg, so the compiler
  // allocates it against that role's register budget
  if (warp >= 12) {
  regs_to<kRegsWg3>();
  dq_readout();
  } else if (warp >= 8) {
  regs_to<kRegsWg2>();
  if (warp == 8) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int gs = 0;  // global step index: stage gs & 1, ring phase (gs >> 1) & 1
      bool ok = true;
      for (int r = 0, uc = 0; ok; ++r) {
        const int ui = unit_index(a.cta_off, r, cta);
        if (ui < 0) break;
        const BwdUnit u = a.units[ui];
        int kmin, kmax;
        pm.range(u.t * kRows, u.t * kRows + kRows, kmin, kmax);
        StepIter<SHARD, NAT> it;
        it.init(pm, u.h * G, u.h * G + G, kmin, a.q_lo, a.q_hi);
        if (!it.begin(pm)) continue;  // every role skips a unit no query sees
        // everything a load needs is computed before the wait that releases
        // its stage: the dO stage is freed late (it stages dQ), and any work
        // between that release and the load lands on the MMA chain
        const int krow = mem_row<NAT>(pm, u.t * kRows);
        asm volatile("" ::"r"(krow));
        if (!(ok = mbar_wait(&bar.kv_empty, (uc & 1) ^ 1, ab))) break;
        mbar_expect_tx(&bar.kv_full, 2 * C::TILE);
        for (int bx = 0; bx < D / 64; ++bx) {
          tma_load_4d(smem + C::OFF_K + bx * kRows * 128, &a.tk, &bar.kv_full, bx * 64, u.h, krow, u.b);
          tma_load_4d(smem + C::OFF_V + bx * kRows * 128, &a.tv, &bar.kv_full, bx * 64, u.h, krow, u.b);
        }
        bool more;
        do {
          const int hq = it.hq, qt = it.qt, qrow = it.mem_row(), qmin = it.qmin(pm);
          more = it.next(pm);  // (the step after this one)
          const int st = gs & 1;
          const uint32_t ph = ((gs >> 1) & 1) ^ 1;
          const size_t vo = ((size_t)u.b * a.sh.Hq + hq) * a.Spad + (size_t)qt * kRows;
          unsigned char* vec = smem + C::OFF_VEC + st * C::VEC_BYTES;
          // (an empty asm that reads the values keeps the compiler from sinking
          // their computation below the waits)
          asm volatile("" ::"r"(qrow), "l"(vo), "r"(it.qt), "r"(it.hq), "r"((int)more), "r"(qmin));
          if (!(ok = mbar_wait(&bar.q_empty[st], ph, ab))) break;
          info[st].hq = hq;
          info[st].qt = qt;
          info[st].last = more ? 0 : 1;
          info[st].qmin = qmin;
          mbar_expect_tx(&bar.q_full[st], C::TILE + C::VEC_BYTES);  // (release: the info is visible to q_full's waiters)
          for (int bx = 0; bx < D / 64; ++bx)
            tma_load_4d(smem + C::OFF_Q + st * C::TILE + bx * kRows * 128, &a.tq, &bar.q_full[st], bx * 64, hq, qrow,
                        u.b);
          bulk_load(vec, a.lse_l2 + vo, kRows * 4, &bar.q_full[st]);
          bulk_load(vec + kRows * 4, a.delta + vo, kRows * 4, &bar.q_full[st]);
          if (!(ok = mbar_wait(&bar.do_empty[st], ph, ab))) break;
          mbar_expect_tx(&bar.do_full[st], C::TILE);
          for (int bx = 0; bx < D / 64; ++bx)
            tma_load_4d(smem + C::OFF_DO + st * C::TILE + bx * kRows * 128, &a.tdo, &bar.do_full[st], bx * 64, hq, qrow,
                        u.b);
          // with the unit's last step queued, the next unit's K and V go to
          // L2: their loads wait for this unit's last MMA, and would otherwise
          // meet the full HBM latency at every unit boundary
          if (!more) {
            const int ui2 = unit_index(a.cta_off, r + 1, cta);
            if (ui2 >= 0) {
              const BwdUnit u2 = a.units[ui2];
              const int krow2 = mem_row<NAT>(pm, u2.t * kRows);
              for (int bx = 0; bx < D / 64; ++bx) {
                tma_prefetch_l2_4d(&a.tk, bx * 64, u2.h, krow2, u2.b);
                tma_prefetch_l2_4d(&a.tv, bx * 64, u2.h, krow2, u2.b);
              }
            }
          }
          ++gs;
        } while (more);
        ++uc;
      }
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t IDESC_S = idesc_bf16(128, kRows, 0, 0);  // S^T, dP^T: K-major x K-major
      constexpr uint32_t IDESC_ACC = idesc_bf16(128, D, 0, 1);    // P^T / dS^T (TMEM) x dO / Q (MN-major)
      constexpr uint32_t IDESC_DQ = idesc_bf16(128, D, 1, 1);     // dS (MN-major) x K (MN-major)
      const uint32_t s0 = smem_u32(smem);
      const uint64_t dK_k = sdesc_sw128(s0 + C::OFF_K, 16, 1024);          // K as K-major A
      const uint64_t dV_k = sdesc_sw128(s0 + C::OFF_V, 16, 1024);          // V as K-major A
      const uint64_t dK_mn = sdesc_sw128(s0 + C::OFF_K, kRows * 128, 1024);  // K as MN-major B
      const uint64_t dS_mn = sdesc_sw128(s0 + C::OFF_DS, kRows * 128, 1024); // dS as MN-major A
      auto kstep = [](int kk) { return (uint64_t)((((kk >> 2) * (kRows * 128)) + (kk & 3) * 32) >> 4); };
      auto issue_s = [&](int st) {
        const uint64_t bq = sdesc_sw128(s0 + C::OFF_Q + st * C::TILE, 16, 1024);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          mma_ss(tmem + C::T_S, dK_k + kstep(kk), bq + kstep(kk), IDESC_S, kk > 0 ? 1u : 0u);
        mma_commit(&bar.s_full);
      };
      auto issue_dp = [&](int st) {
        const uint64_t bo = sdesc_sw128(s0 + C::OFF_DO + st * C::TILE, 16, 1024);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          mma_ss(tmem + C::T_DP, dV_k + kstep(kk), bo + kstep(kk), IDESC_S, kk > 0 ? 1u : 0u);
        mma_commit(&bar.dp_full);
      };
      auto issue_dv = [&](int st, bool acc) {
        const uint64_t bo = sdesc_sw128(s0 + C::OFF_DO + st * C::TILE, kRows * 128, 1024);
#pragma unroll
        for (int kk = 0; kk < kRows / 16; ++kk)
          mma_ts(tmem + C::T_DV, tmem + C::T_S + packed_col<64>(kk * 16), bo + ((kk * 16 * 128) >> 4), IDESC_ACC,
                 (acc || kk > 0) ? 1u : 0u);
      };
      auto issue_dk = [&](int st, bool acc) {
        const uint64_t bq = sdesc_sw128(s0 + C::OFF_Q + st * C::TILE, kRows * 128, 1024);
#pragma unroll
        for (int kk = 0; kk < kRows / 16; ++kk)
          mma_ts(tmem + C::T_DK, tmem + C::T_DP + packed_col<64>(kk * 16), bq + ((kk * 16 * 128) >> 4), IDESC_ACC,
                 (acc || kk > 0) ? 1u : 0u);
      };
      auto issue_dq = [&]() {
#pragma unroll
        for (int kk = 0; kk < kRows / 16; ++kk)
          mma_ss(tmem + C::T_DP, dS_mn + ((kk * 16 * 128) >> 4), dK_mn + ((kk * 16 * 128) >> 4), IDESC_DQ,
                 kk > 0 ? 1u : 0u);
        mma_commit(&bar.dq_full);
      };

      int gs = 0;
      bool ok = true;
      for (int r = 0, uc = 0; ok; ++r) {
        const int ui = unit_index(a.cta_off, r, cta);
        if (ui < 0) break;
        const BwdUnit u = a.units[ui];
        int kmin, kmax;
        pm.range(u.t * kRows, u.t * kRows + kRows, kmin, kmax);
        StepIter<SHARD, NAT> it;
        it.init(pm, u.h * G, u.h * G + G, kmin, a.q_lo, a.q_hi);
        if (!it.begin(pm)) continue;
        if (!(ok = mbar_wait(&bar.kv_full, uc & 1, ab))) break;
        tc_fence_after();
        // prologue: S and dP of the unit's first step
        if (!(ok = mbar_wait(&bar.q_full[gs & 1], (gs >> 1) & 1, ab))) break;
        tc_fence_after();
        bool more = !info[gs & 1].last;
        issue_s(gs & 1);
        if (gs > 0 && !(ok = mbar_wait(&bar.dq_free, (gs - 1) & 1, ab))) break;  // dQ of the last step read out
        if (!(ok = mbar_wait(&bar.do_full[gs & 1], (gs >> 1) & 1, ab))) break;
        tc_fence_after();
        issue_dp(gs & 1);
        for (int j = 0; ok; ++j, ++gs) {
          const int st = gs & 1;
          const bool this_more = more;
          if (!(ok = mbar_wait(&bar.p_full, gs & 1, ab))) break;
          tc_fence_after();
          issue_dv(st, j > 0);
          if (this_more) {
            if (!(ok = mbar_wait(&bar.q_full[st ^ 1], ((gs + 1) >> 1) & 1, ab))) break;
            tc_fence_after();
            more = !info[st ^ 1].last;
            issue_s(st ^ 1);
          }
          if (!(ok = mbar_wait(&bar.dst_full, gs & 1, ab))) break;
          tc_fence_after();
          issue_dk(st, j > 0);
          mma_commit(&bar.q_empty[st]);  // Q_j (S_j, dK_j) and its vectors are done
          if (!(ok = mbar_wait(&bar.dss_full, gs & 1, ab))) break;
          tc_fence_after();
          issue_dq();
          if (!this_more) break;
          if (!(ok = mbar_wait(&bar.dq_free, gs & 1, ab))) break;
          if (!(ok = mbar_wait(&bar.do_full[st ^ 1], ((gs + 1) >> 1) & 1, ab))) break;
          tc_fence_after();
          issue_dp(st ^ 1);
        }
        if (!ok) break;
        ++gs;
        mma_commit(&bar.acc_full);
        mma_commit(&bar.kv_empty);  // K (last read by dQ) and V are done
        ++uc;
      }
      mma_drain(&bar.done, a.err);
    }
  } else if (warp == 10) {
    // ------------------------------------------------------------ dQ reducer
    // adds each staged dQ tile into the fp32 accumulator; the boxes in the dS
    // space go first, in their own bulk group, because the next dS waits on them.
    // The accumulator is in slot order for natural-order tensors too (the
    // rounding pass writes each slot's row to its natural row): measured on
    // the Llama3.1-70B-shaped layer, reduce-adds into the natural rows cost
    // the natural-order backward about a fifth of its time, into the slot
    // rows nothing measurable, for the same tiles in the same order.
    if (lane == 0) {
      int gs = 0;
      for (int r = 0;; ++r) {
        const int ui = unit_index(a.cta_off, r, cta);
        if (ui < 0) break;
        const BwdUnit u = a.units[ui];
        int kmin, kmax;
        pm.range(u.t * kRows, u.t * kRows + kRows, kmin, kmax);
        StepIter<SHARD, NAT> it;
        it.init(pm, u.h * G, u.h * G + G, kmin, a.q_lo, a.q_hi);
        if (!it.begin(pm)) continue;
        do {
          const int hq = it.hq, qt = it.qt;
          // runs on after an abort: the staging is garbage, the waits bounded
          mbar_wait(C::NBOX > 2 ? &bar.staged_ds : &bar.staged, gs & 1, ab);
#pragma unroll
          for (int box = 0; box < C::NBOX; ++box) {
            if (box == 2) mbar_wait(&bar.staged, gs & 1, ab);
            const unsigned char* bb = box < 2 ? smem + C::OFF_DS + box * (kRows * 128)
                                              : smem + C::OFF_DO + (gs & 1) * C::TILE + (box - 2) * (kRows * 128);
            tma_reduce_add_4d(bb, &a.tdq, box * 32, hq, qt * kRows, u.b);  // slot order (see above)
            if (box == 1) bulk_commit_group();
          }
          if (C::NBOX > 2) {
            bulk_commit_group();
            bulk_wait_read<1>();
          } else {
            bulk_wait_read<0>();
          }
          mbar_arrive(&bar.ds_free);  // the dS tile (staging space) may be rewritten
          bulk_wait_read<0>();
          mbar_arrive(&bar.do_empty[gs & 1]);  // the dO stage (staging space) may be reloaded
          ++gs;
        } while (it.next(pm));
      }
      bulk_wait_all();  // every dQ reduce has landed before the CTA retires
    }
  }
  } else {
    regs_to<kRegsEw>();
    // ------------------------------------------------------------ element-wise warps
    // Group g (warps 4g..4g+3) owns query columns [64g, 64g+64) of S^T/dP^T
    // (thread = key row = TMEM lane) and, at the end of a unit, dV/dK columns
    // [gD/2, (g+1)D/2).  A failed wait (abort or timeout) runs on with whatever
    // is in TMEM, so every role walks all of its steps and every wait stays
    // bounded.
    const int g = warp >> 2;
    const int row = ((warp & 3) << 5) + lane;  // TMEM lane
    const uint32_t lane_base = uint32_t((warp & 3) * 32) << 16;
    const uint64_t sl2x2 = f2pack(a.scale_log2, a.scale_log2);
    int gs = 0;

    // the next unit's descriptor is fetched while this unit's dK/dV go out
    // (pf: the unit index r it belongs to, -2 past the CTA's last unit)
    int pf = -1;
    BwdUnit un{};
    for (int r = 0, uc = 0;; ++r) {
      BwdUnit u;
      if (pf == r) {
        u = un;
      } else {
        if (pf == -2) break;
        const int ui = unit_index(a.cta_off, r, cta);
        if (ui < 0) break;
        u = a.units[ui];
      }
      pf = -1;
      const int kslot = u.t * kRows + row;
      const bool kvalid = kslot < pm.S;
      const int kpos = kvalid ? pm.pos(kslot) : 0x7fffffff;
      int kmin, kmax;
      pm.range(u.t * kRows, u.t * kRows + kRows, kmin, kmax);
      const bool k_inside = u.t * kRows + kRows <= pm.S;
      {
        StepIter<SHARD, NAT> it;
        it.init(pm, u.h * G, u.h * G + G, kmin, a.q_lo, a.q_hi);
        if (!it.begin(pm)) continue;
      }
      bool last;
      do {
        const int st = gs & 1;
        // ---- P into TMEM as bf16 (fp32 copy kept for dS)
        mbar_wait(&bar.s_full, gs & 1, ab);
        mbar_wait(&bar.q_full[st], (gs >> 1) & 1, ab);
        tc_fence_after();
        const int qt = info[st].qt;
        last = info[st].last != 0;
        const int qmin = info[st].qmin;  // (from the producer: no division on this path)
        const float* lse_s = reinterpret_cast<const float*>(smem + C::OFF_VEC + st * C::VEC_BYTES) + g * 64;
        const float* del_s = lse_s + kRows;
        float p[64];
        const uint32_t t_s = tmem + lane_base + C::T_S + g * 64;
        const uint32_t t_pk = tmem + lane_base + C::T_S + packed_col<64>(g * 64);
        const bool q_inside = !SHARD || (qt * kRows >= a.q_lo && qt * kRows + kRows <= a.q_hi);
        if ((kmax <= qmin) && k_inside && q_inside)
          ew_p<false, SHARD>(t_s, t_pk, lse_s, sl2x2, p, kpos, pm, 0, 0, 0);
        else
          ew_p<true, SHARD>(t_s, t_pk, lse_s, sl2x2, p, kpos, pm, qt * kRows + g * 64, a.q_lo, a.q_hi);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&bar.p_full);
        // ---- dS = P * (dP - D): bf16 into TMEM (for dK), then shared memory (for dQ)
        mbar_wait(&bar.dp_full, gs & 1, ab);
        tc_fence_after();
        uint32_t dp[2][32], dk[2][16];
        tmem_ld32(tmem + lane_base + C::T_DP + g * 64, dp[0]);
        tmem_ld32(tmem + lane_base + C::T_DP + g * 64 + 32, dp[1]);
        tmem_ld_wait();
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const uint64_t* nd2 = reinterpret_cast<const uint64_t*>(del_s + 32 * h);
#pragma unroll
          for (int c = 0; c < 32; c += 2) {
            float d0, d1;
            f2unpack(f2mul(f2pack(p[32 * h + c], p[32 * h + c + 1]), f2add(f2pack_u(dp[h][c], dp[h][c + 1]), nd2[c >> 1])),
                     d0, d1);
            dk[h][c >> 1] = pack_bf16(d0, d1);
          }
          tmem_st16(tmem + lane_base + C::T_DP + packed_col<64>(g * 64 + 32 * h), dk[h]);
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&bar.dst_full);
        if (gs > 0) mbar_wait(&bar.ds_free, (gs - 1) & 1, ab);  // the previous dQ tile left the dS space
        unsigned char* dsr = smem + C::OFF_DS + g * (kRows * 128) + row * 128;  // this key row of query half g
#pragma unroll
        for (int chunk = 0; chunk < 8; ++chunk)  // 8 query columns per 16-byte chunk
          *reinterpret_cast<uint4*>(dsr + ((chunk ^ (row & 7)) << 4)) =
              make_uint4(dk[chunk >> 2][4 * (chunk & 3)], dk[chunk >> 2][4 * (chunk & 3) + 1],
                         dk[chunk >> 2][4 * (chunk & 3) + 2], dk[chunk >> 2][4 * (chunk & 3) + 3]);
        fence_proxy_async_smem();
        mbar_arrive(&bar.dss_full);
        ++gs;
      } while (!last);
      if constexpr (!SHARD) {  // (in the per-shard kernel it cost registers and 2% of its time)
        const int ui2 = unit_index(a.cta_off, r + 1, cta);
        if (ui2 >= 0) {
          un = a.units[ui2];
          pf = r + 1;
        } else {
          pf = -2;
        }
      }
      // dV and scale*dK of this key tile
      mbar_wait(&bar.acc_full, uc & 1, ab);
      tc_fence_after();
      if constexpr (SHARD) {  // one shard's backward also writes unrounded fp32 partials (staged
        // through the dS space half by half like the bf16 path below, they took 3% longer)
        const size_t orow = ((size_t)u.b * pm.S + (kvalid ? mem_row<NAT>(pm, kslot) : 0)) * a.sh.Hkv + u.h;
        const float sc = a.scale;
#pragma unroll
        for (int which = 0; which < 2; ++which) {
          const float f = which ? sc : 1.f;
          __nv_bfloat16* dst0 = static_cast<__nv_bfloat16*>(which ? a.dk : a.dv);
          float* part0 = which ? a.dk_part : a.dv_part;
#pragma unroll 1
          for (int c0 = g * (D / 2); c0 < (g + 1) * (D / 2); c0 += 32) {
            uint32_t o[32];
            tmem_ld32(tmem + lane_base + (which ? C::T_DK : C::T_DV) + c0, o);
            tmem_ld_wait();
            if (kvalid && (!SHARD || dst0)) {
              uint4* dst = reinterpret_cast<uint4*>(dst0 + orow * D + c0);
#pragma unroll
              for (int v4 = 0; v4 < 4; ++v4)
                dst[v4] = make_uint4(pack_bf16(f * __uint_as_float(o[8 * v4 + 0]), f * __uint_as_float(o[8 * v4 + 1])),
                                     pack_bf16(f * __uint_as_float(o[8 * v4 + 2]), f * __uint_as_float(o[8 * v4 + 3])),
                                     pack_bf16(f * __uint_as_float(o[8 * v4 + 4]), f * __uint_as_float(o[8 * v4 + 5])),
                                     pack_bf16(f * __uint_as_float(o[8 * v4 + 6]), f * __uint_as_float(o[8 * v4 + 7])));
            }
            if (SHARD && kvalid) {  // per-shard partial, unrounded
              float4* dst = reinterpret_cast<float4*>(part0 + orow * D + c0);
#pragma unroll
              for (int v4 = 0; v4 < 8; ++v4)
                dst[v4] = make_float4(f * __uint_as_float(o[4 * v4 + 0]), f * __uint_as_float(o[4 * v4 + 1]),
                                      f * __uint_as_float(o[4 * v4 + 2]), f * __uint_as_float(o[4 * v4 + 3]));
            }
          }
        }
      } else {
        // through the dS space (free once the last step's dQ tile has been
        // reduced), so that each warp store writes whole lines: a thread
        // stores its key row's half in bf16 (16-byte pieces, XOR-swizzled by
        // row), then the 256 threads read the tile back row by row.  Stored
        // straight from the TMEM rows instead, every warp store touched 32
        // lines 16 bytes at a time and the epilogue took about 8,000 clocks
        // (now about 6,000, a third of it the wait for the dS space).
        // Writing dK/dV from the dQ read-out warps instead, so that these
        // warps went straight on to the next unit, shortened the unit
        // boundary but made every step about 4% slower.
        mbar_wait(&bar.ds_free, (gs - 1) & 1, ab);
        int* mrow_s = reinterpret_cast<int*>(smem + C::OFF_MROW);
        if (g == 0) mrow_s[row] = kvalid ? mem_row<NAT>(pm, kslot) : -1;
        constexpr int KC = D / 8;  // 16-byte pieces of a row
        unsigned char* const stg = smem + C::OFF_DS;
        const size_t rbase = (size_t)u.b * pm.S;
        const int tid_ew = (warp << 5) + lane;
#pragma unroll
        for (int which = 0; which < 2; ++which) {
          const float f = which ? a.scale : 1.f;
          uint32_t o[2][32];
          tmem_ld32(tmem + lane_base + (which ? C::T_DK : C::T_DV) + g * (D / 2), o[0]);
          if (D / 2 > 32) tmem_ld32(tmem + lane_base + (which ? C::T_DK : C::T_DV) + g * (D / 2) + 32, o[1]);
          tmem_ld_wait();
          unsigned char* sr = stg + row * (D * 2);
#pragma unroll
          for (int j = 0; j < KC / 2; ++j) {  // piece k = columns 8k..8k+7
            const int k = g * (KC / 2) + j;
            const uint32_t* x = &o[j >> 2][8 * (j & 3)];
            *reinterpret_cast<uint4*>(sr + ((k ^ (row & 7)) << 4)) =
                make_uint4(pack_bf16(f * __uint_as_float(x[0]), f * __uint_as_float(x[1])),
                           pack_bf16(f * __uint_as_float(x[2]), f * __uint_as_float(x[3])),
                           pack_bf16(f * __uint_as_float(x[4]), f * __uint_as_float(x[5])),
                           pack_bf16(f * __uint_as_float(x[6]), f * __uint_as_float(x[7])));
          }
          named_bar(1, 256);
          __nv_bfloat16* dst0 = static_cast<__nv_bfloat16*>(which ? a.dk : a.dv);
#pragma unroll
          for (int i = 0; i < KC / 2; ++i) {
            const int pc = tid_ew + 256 * i, rr = pc / KC, k = pc % KC;
            const int mr = mrow_s[rr];
            if (mr >= 0)
              *reinterpret_cast<uint4*>(dst0 + ((rbase + mr) * a.sh.Hkv + u.h) * D + 8 * k) =
                  *reinterpret_cast<const uint4*>(stg + rr * (D * 2) + ((k ^ (rr & 7)) << 4));
          }
          named_bar(1, 256);  // the tile is read back: the space takes dK, then the next unit's dS
        }
      }
      tc_fence_before();
      ++uc;
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

// dq (bf16, [B, S, Hq, D]) = scale * the fp32 accumulator; 8 elements per thread
__global__ void __launch_bounds__(256) bwd_dq_round_kernel(const float* __restrict__ acc, __nv_bfloat16* dq, long long n8,
                                                           float scale) {
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n8; i += (long long)gridDim.x * blockDim.x) {
    const float4 x = __ldcs(reinterpret_cast<const float4*>(acc) + 2 * i);
    const float4 y = __ldcs(reinterpret_cast<const float4*>(acc) + 2 * i + 1);
    reinterpret_cast<uint4*>(dq)[i] =
        make_uint4(pack_bf16(scale * x.x, scale * x.y), pack_bf16(scale * x.z, scale * x.w),
                   pack_bf16(scale * y.x, scale * y.y), pack_bf16(scale * y.z, scale * y.w));
  }
}

// natural-order dq: row b*S + pos(s) of dq = scale * row b*S + s of the
// slot-order accumulator; one row (Hq*D elements) per CTA iteration
__global__ void __launch_bounds__(256) bwd_dq_round_nat_kernel(const float* __restrict__ acc, __nv_bfloat16* dq,
                                                               int B, PosMap pm, int row8, float scale) {
  for (long long r = blockIdx.x; r < (long long)B * pm.S; r += gridDim.x) {
    const int b = int(r / pm.S), s = int(r - (long long)b * pm.S);
    const float4* src = reinterpret_cast<const float4*>(acc) + 2 * r * row8;
    uint4* dst = reinterpret_cast<uint4*>(dq) + ((long long)b * pm.S + pm.pos(s)) * row8;
    for (int i = threadIdx.x; i < row8; i += blockDim.x) {
      const float4 x = __ldcs(src + 2 * i);
      const float4 y = __ldcs(src + 2 * i + 1);
      dst[i] = make_uint4(pack_bf16(scale * x.x, scale * x.y), pack_bf16(scale * x.z, scale * x.w),
                          pack_bf16(scale * y.x, scale * y.y), pack_bf16(scale * y.z, scale * y.w));
    }
  }
}

template <int D, bool SHARD, bool NAT>
cudaError_t launch_fused(const BwdArgs& a, int grid, cudaStream_t st) {
  auto kern = attn_bwd_fused_kernel<D, SHARD, NAT>;
  // more than half of an SM's shared memory: one CTA per SM, so the CTA's
  // 512-column TMEM allocation never waits for a neighbour
  int smem = FCfg<D>::SMEM;
  if (smem < 120 * 1024) smem = 120 * 1024;
  // setmaxnreg.inc only succeeds if the launch reserved kRegsLaunchF per thread
  cudaFuncAttributes fa0;
  cudaError_t e = cudaFuncGetAttributes(&fa0, kern);
  if (e != cudaSuccess) return e;
  if (fa0.numRegs != kRegsLaunchF) return cudaErrorInvalidConfiguration;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  kern<<<grid, kThreadsF, smem, st>>>(a);
  e = cudaGetLastError();
  if (e != cudaSuccess) {
    cudaFuncAttributes fa{};
    cudaFuncGetAttributes(&fa, kern);
    fprintf(stderr, "attn_bwd_fused<%d>: %s (regs %d, max threads %d, smem %d)\n", D, cudaGetErrorString(e),
            fa.numRegs, fa.maxThreadsPerBlock, smem);
  }
  return e;
}

}  // namespace

bool bwd_fused_supported(int Dqk, int Dv) { return Dqk == Dv && (Dqk == 64 || Dqk == 128); }

cudaError_t launch_attn_bwd_fused(const BwdArgs& a, int grid, cudaStream_t st) {
  const bool shard = a.dk_part != nullptr;  // (the per-shard call does not take natural-order tensors)
  const bool nat = PosMap::make(a.sh.S, a.sh.cp, a.sh.lb).lb == 2;
  if (a.sh.Dqk == 64) {
    if (shard) return launch_fused<64, true, false>(a, grid, st);
    return nat ? launch_fused<64, false, true>(a, grid, st) : launch_fused<64, false, false>(a, grid, st);
  }
  if (shard) return launch_fused<128, true, false>(a, grid, st);
  return nat ? launch_fused<128, false, true>(a, grid, st) : launch_fused<128, false, false>(a, grid, st);
}

cudaError_t launch_bwd_dq_round_nat(const float* acc, void* dq, const AttnShape& sh, float scale, cudaStream_t st) {
  const PosMap pm = PosMap::make(sh.S, sh.cp, sh.lb);
  long long blocks = (long long)sh.B * sh.S;
  if (blocks > 152LL * 16) blocks = 152LL * 16;
  bwd_dq_round_nat_kernel<<<(int)blocks, 256, 0, st>>>(acc, static_cast<__nv_bfloat16*>(dq), sh.B, pm,
                                                       sh.Hq * sh.Dqk / 8, scale);
  return cudaGetLastError();
}

cudaError_t launch_bwd_dq_round(const float* acc, void* dq, long long n, float scale, cudaStream_t st) {
  const long long n8 = n / 8;  // n is a multiple of 64 (head dim)
  long long blocks = (n8 + 255) / 256;
  if (blocks > 152LL * 16) blocks = 152LL * 16;
  bwd_dq_round_kernel<<<(int)blocks, 256, 0, st>>>(acc, static_cast<__nv_bfloat16*>(dq), n8, scale);
  return cudaGetLastError();
}

}  // namespace cpattn
