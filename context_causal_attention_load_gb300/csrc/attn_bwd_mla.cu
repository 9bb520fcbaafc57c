// Fused flash backward for MLA head dims (query/key 192 = 128 nope + 64 rope,
// value 128).
//
// Same gradient as the other backward kernels (the textbook gradient of
// out = softmax(scale q k^T + mask) v under the reordered causal mask, "Add
// support for EP to context parallelism in self-attention", Main code changes:
// MLA under context parallelism), in one pass like the equal-dims fused
// kernel: a CTA owns a 128-row key tile of one KV head and walks every (query
// head of the group, 128-row query tile) that sees it, each tile as two
// 64-row half-steps.  Per half-step, on tcgen05:
//   S^T  = K Q^T    (128 key lanes x 64)  -> P^T  (bf16, in place)
//   dP^T = V dO^T   (128 key lanes x 64)  -> dS^T (bf16, in place) and
//                                            dS^T (bf16, shared memory)
//   dV += P^T dO (N = 128),  dK += dS^T Q (N = 192)   (TMEM accumulators)
//   dQ^T = K^T dS^T: the step's dQ transposed, dims as the MMA rows, in two
//          MMAs of 128 rows: dims 0-127 into dP's columns and dims 64-191
//          into a 64-column block of its own (dims 64-127 come out twice;
//          the read-out keeps the first copy)
// dQ^T is staged in shared memory as fp32 query rows and added into the fp32
// dQ accumulator by TMA reduce-add; the rounding pass applies the softmax
// scale.  S and dP are formed once per (key, query) pair, not twice as in the
// two-kernel path.
//
// 64-row half-steps keep TMEM within 512 columns: S 64 | dP (and dQ dims
// 0-127) 64 | dQ dims 64-191 64 | dV 128 | dK 192.  MMA order per half-step
// j: dP_j, dV_j, S_{j+1}, dK_j, dQ_j; the element-wise warps form P_{j+1}
// while dK_j and dQ_j execute.  A warpgroup of its own reads dQ_j out of TMEM
// the moment it is complete (dP_{j+1} needs its columns) and stages it; a
// reducer thread adds the staged tile into the accumulator.
//
// Shared memory (226 KiB): K (48 KiB) and V (32 KiB) tiles resident per
// unit, two stages of Q (24 KiB) and dO (16 KiB) half-tiles with their -lse
// and -D vectors, the dS^T tile (16 KiB) and the fp32 dQ staging (48 KiB).
#include <cstdio>

#include "common.cuh"
#include "internal.h"

namespace cpattn {
namespace {

// warps 0-7 element-wise (two 32-column groups), 8 TMA producer, 9 MMA
// issuer, 10 dQ reducer, 11 idle, 12-15 dQ read-out
constexpr int kThreadsM = 512;
constexpr int kKeys = 128;  // key rows per unit; query rows per tile of the walk
constexpr int kHalf = 64;   // query rows per half-step
constexpr int kDqk = 192, kDv = 128;

struct MCfg {
  static constexpr int K_BYTES = kKeys * kDqk * 2;  // 3 boxes of 128 rows x 128 B
  static constexpr int V_BYTES = kKeys * kDv * 2;   // 2 boxes
  static constexpr int KBOX = kKeys * 128;          // 16 KiB
  static constexpr int QBOX = kHalf * 128;          // 8 KiB
  static constexpr int Q_BYTES = 3 * QBOX;          // a half-step's Q rows
  static constexpr int DO_BYTES = 2 * QBOX;         // its dO rows
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = OFF_K + K_BYTES;
  static constexpr int OFF_Q = OFF_V + V_BYTES;     // stage s at OFF_Q + s*Q_BYTES
  static constexpr int OFF_DO = OFF_Q + 2 * Q_BYTES;
  static constexpr int OFF_DS = OFF_DO + 2 * DO_BYTES;  // dS^T: 128 key rows x 64 queries (bf16)
  static constexpr int DS_BYTES = kKeys * 128;
  static constexpr int OFF_STG = OFF_DS + DS_BYTES;     // dQ staging: 6 boxes of 64 query rows x 32 fp32
  static constexpr int STG_BOX = kHalf * 128;
  static constexpr int OFF_VEC = OFF_STG + 6 * STG_BOX;  // stage s: -lse*log2e[64], then -D[64] (fp32)
  static constexpr int VEC_BYTES = 2 * kHalf * 4;
  static constexpr int OFF_BAR = OFF_VEC + 2 * VEC_BYTES;
  static constexpr int OFF_MISC = OFF_BAR + 256;  // TMEM address, abort flag, MStepInfo[2] at +32
  static constexpr int SMEM = OFF_MISC + 80;
  static_assert(SMEM <= 232448, "shared memory budget");
  static_assert(OFF_V % 1024 == 0 && OFF_Q % 1024 == 0 && OFF_DO % 1024 == 0 && OFF_DS % 1024 == 0 &&
                    OFF_STG % 1024 == 0 && Q_BYTES % 1024 == 0 && DO_BYTES % 1024 == 0,
                "swizzled tiles need 1024-byte alignment");
  // TMEM columns
  static constexpr int T_S = 0;
  static constexpr int T_DP = 64;    // dP^T / dS^T, then dQ^T dims 0-127
  static constexpr int T_DQ1 = 128;  // dQ^T dims 64-191
  static constexpr int T_DV = 192;
  static constexpr int T_DK = 320;
  static_assert(T_DK + kDqk == 512, "TMEM budget");
};

// what the producer publishes with each Q stage
struct MStepInfo {
  int hq, qt, half, last, qmin;  // qmin: first position of the half-step's rows (decides the masked path)
};

struct MBars {
  uint64_t kv_full, kv_empty;
  uint64_t q_full[2], q_empty[2], do_full[2], do_empty[2];
  uint64_t s_full, p_full, dp_full, dst_full, dss_full, ds_free, dq_full, dq_free, dq1_free, staged, stg_free;
  uint64_t acc_full, done;
};
static_assert(sizeof(MBars) <= 256, "barrier area");

// (query head, 128-row query tile) steps of a key-tile unit, walked from the
// top of the sequence down by position where every tile of slots is one tile
// of positions (see the equal-dims fused kernel), else in slot order
template <bool NAT>
struct MStepIter {
  int h_end, kmin;
  bool posw;
  int tpc, first, top;
  int hq, qt, pt, ch, off;

  __device__ __forceinline__ void init(const PosMap& pm, int h0, int h_end_, int kmin_) {
    h_end = h_end_;
    kmin = kmin_;
    hq = h0;
    posw = NAT || pm.lb == 0 || pm.c % kKeys == 0;
    tpc = pm.lb ? pm.c / kKeys : 1;
    first = kmin / kKeys;
    top = (pm.S + kKeys - 1) / kKeys - 1;
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
  __device__ __forceinline__ bool begin(const PosMap& pm) {
    if (posw) {
      to_top(pm);
      return true;
    }
    for (;;) {
      qt = next_q_tile(pm, kKeys, -1, kmin);
      if (qt >= 0) return true;
      if (++hq >= h_end) return false;
    }
  }
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
    qt = next_q_tile(pm, kKeys, qt, kmin);
    if (qt >= 0) return true;
    if (++hq >= h_end) return false;
    qt = next_q_tile(pm, kKeys, -1, kmin);
    return qt >= 0;
  }
  // memory row of the current query tile
  __device__ __forceinline__ int mem_row() const { return NAT ? pt * kKeys : qt * kKeys; }
  // first position of the current tile's rows [half * kHalf, +kHalf)
  __device__ __forceinline__ int qmin(const PosMap& pm, int half) const {
    if (posw) return pt * kKeys + half * kHalf;
    int mn, mx;
    pm.range(qt * kKeys + half * kHalf, qt * kKeys + half * kHalf + kHalf, mn, mx);
    return mn;
  }
};

template <bool NAT>
__device__ __forceinline__ int mla_mem_row(const PosMap& pm, int slot) { return NAT ? pm.pos(slot) : slot; }

// P for this thread's 32 query columns of a half-step: scores from TMEM (t_s),
// p = exp2(s * scale*log2e - lse*log2e), zeroed where the key's position is
// past the query's (MASKED only; positions walked slot by slot from slot0),
// kept in fp32 for dS and stored back to TMEM (t_pk) as packed bf16
template <bool MASKED>
__device__ __forceinline__ void mla_ew_p(uint32_t t_s, uint32_t t_pk, const float* lse_s, uint64_t sl2x2,
                                         float (&p)[32], int kpos, const PosMap& pm, int slot0) {
  int ck = 0, ct = 0, cbase = 0;
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
    return q;
  };
  uint32_t sv[32];
  tmem_ld32(t_s, sv);
  tmem_ld_wait();
  const uint64_t* nl2 = reinterpret_cast<const uint64_t*>(lse_s);
  uint32_t pk[16];
#pragma unroll
  for (int c = 0; c < 32; c += 2) {
    float p0, p1;
    f2unpack(f2fma(f2pack_u(sv[c], sv[c + 1]), sl2x2, nl2[c >> 1]), p0, p1);
    p0 = fast_exp2(p0);
    p1 = fast_exp2(p1);
    if (MASKED) {
      const int q0 = next_qpos(slot0 + c);
      const int q1 = next_qpos(slot0 + c + 1);
      p0 = kpos <= q0 ? p0 : 0.f;
      p1 = kpos <= q1 ? p1 : 0.f;
    }
    p[c] = p0;
    p[c + 1] = p1;
    pk[c >> 1] = pack_bf16(p0, p1);
  }
  tmem_st16(t_pk, pk);
}

// fire-and-forget fp32 add of four consecutive floats (16-byte aligned) in global memory
__device__ __forceinline__ void mla_red_add_v4(float* p, float x, float y, float z, float w) {
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(x), "f"(y), "f"(z), "f"(w) : "memory");
}

// this thread's bulk async-groups, all but the newest N, have read their sources
template <int N>
__device__ __forceinline__ void mla_bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

// NAT: tensors in natural order (zero-copy load balance); the dQ accumulator
// stays in slot order and the rounding pass writes each slot's row to its
// natural row
template <bool NAT>
__global__ void __launch_bounds__(kThreadsM, 1) attn_bwd_mla_kernel(const __grid_constant__ BwdArgs a) {
  using C = MCfg;
  extern __shared__ __align__(1024) unsigned char smem[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (smem_u32(smem) & 1023u) {  // every offset assumes a 1024-byte aligned base
    if (tid == 0) atomicExch(a.err, DEV_SMEM_ALIGN);
    return;
  }
  MBars& bar = *reinterpret_cast<MBars*>(smem + C::OFF_BAR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 16);
  volatile MStepInfo* info = reinterpret_cast<volatile MStepInfo*>(smem + C::OFF_MISC + 32);
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
    mbar_init(&bar.ds_free, 1);
    mbar_init(&bar.dq_full, 1);
    mbar_init(&bar.dq_free, 128);
    mbar_init(&bar.dq1_free, 128);
    mbar_init(&bar.staged, 128);
    mbar_init(&bar.stg_free, 1);
    mbar_init(&bar.acc_full, 1);
    mbar_init(&bar.done, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 9) { tmem_alloc(tmem_slot, 512); tmem_relinquish(); }
  if (warp == 8 && lane == 0) {
    prefetch_tmap(&a.tq); prefetch_tmap(&a.tk); prefetch_tmap(&a.tv); prefetch_tmap(&a.tdo); prefetch_tmap(&a.tdq);
    if (a.rope_shared) prefetch_tmap(&a.tkr);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 8) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int gs = 0;  // global half-step: stage gs & 1, ring phase (gs >> 1) & 1
      bool ok = true;
      for (int r = 0, uc = 0; ok; ++r) {
        const int ui = unit_index(a.cta_off, r, cta);
        if (ui < 0) break;
        const BwdUnit u = a.units[ui];
        int kmin, kmax;
        pm.range(u.t * kKeys, u.t * kKeys + kKeys, kmin, kmax);
        MStepIter<NAT> it;
        it.init(pm, u.h * G, u.h * G + G, kmin);
        if (!it.begin(pm)) continue;  // every role skips a unit no query sees
        const int krow = mla_mem_row<NAT>(pm, u.t * kKeys);
        asm volatile("" ::"r"(krow));
        if (!(ok = mbar_wait(&bar.kv_empty, (uc & 1) ^ 1, ab))) break;
        mbar_expect_tx(&bar.kv_full, C::K_BYTES + C::V_BYTES);
        for (int bx = 0; bx < 3; ++bx) {
          if (bx == 2 && a.rope_shared)  // the rope keys shared by the heads
            tma_load_4d(smem + C::OFF_K + bx * C::KBOX, &a.tkr, &bar.kv_full, 0, 0, krow, u.b);
          else
            tma_load_4d(smem + C::OFF_K + bx * C::KBOX, &a.tk, &bar.kv_full, bx * 64, u.h, krow, u.b);
        }
        for (int bx = 0; bx < 2; ++bx)
          tma_load_4d(smem + C::OFF_V + bx * C::KBOX, &a.tv, &bar.kv_full, bx * 64, u.h, krow, u.b);
        bool more;
        do {
          const int hq = it.hq, qt = it.qt, qrow = it.mem_row();
          const int qmin0 = it.qmin(pm, 0), qmin1 = it.qmin(pm, 1);
          more = it.next(pm);
          for (int half = 0; half < 2 && ok; ++half) {
            const int st = gs & 1;
            const uint32_t ph = ((gs >> 1) & 1) ^ 1;
            const size_t vo = ((size_t)u.b * a.sh.Hq + hq) * a.Spad + (size_t)qt * kKeys + half * kHalf;
            unsigned char* vec = smem + C::OFF_VEC + st * C::VEC_BYTES;
            asm volatile("" ::"r"(qrow), "l"(vo), "r"((int)more));
            if (!(ok = mbar_wait(&bar.q_empty[st], ph, ab))) break;
            info[st].hq = hq;
            info[st].qt = qt;
            info[st].half = half;
            info[st].last = (!more && half == 1) ? 1 : 0;
            info[st].qmin = half ? qmin1 : qmin0;
            mbar_expect_tx(&bar.q_full[st], C::Q_BYTES + C::VEC_BYTES);  // (release: the info is visible to q_full's waiters)
            for (int bx = 0; bx < 3; ++bx)
              tma_load_4d(smem + C::OFF_Q + st * C::Q_BYTES + bx * C::QBOX, &a.tq, &bar.q_full[st], bx * 64, hq,
                          qrow + half * kHalf, u.b);
            bulk_load(vec, a.lse_l2 + vo, kHalf * 4, &bar.q_full[st]);
            bulk_load(vec + kHalf * 4, a.delta + vo, kHalf * 4, &bar.q_full[st]);
            if (!(ok = mbar_wait(&bar.do_empty[st], ph, ab))) break;
            mbar_expect_tx(&bar.do_full[st], C::DO_BYTES);
            for (int bx = 0; bx < 2; ++bx)
              tma_load_4d(smem + C::OFF_DO + st * C::DO_BYTES + bx * C::QBOX, &a.tdo, &bar.do_full[st], bx * 64, hq,
                          qrow + half * kHalf, u.b);
            ++gs;
          }
        } while (more && ok);
        ++uc;
      }
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t IDESC_S = idesc_bf16(128, kHalf, 0, 0);   // S^T, dP^T: K-major x K-major
      constexpr uint32_t IDESC_DV = idesc_bf16(128, kDv, 0, 1);    // P^T (TMEM) x dO (MN-major)
      constexpr uint32_t IDESC_DK = idesc_bf16(128, kDqk, 0, 1);   // dS^T (TMEM) x Q (MN-major)
      constexpr uint32_t IDESC_DQ = idesc_bf16(128, kHalf, 1, 1);  // K^T (MN-major) x dS^T (MN-major)
      const uint32_t s0 = smem_u32(smem);
      const uint64_t dK_k = sdesc_sw128(s0 + C::OFF_K, 16, 1024);  // K as K-major A
      const uint64_t dV_k = sdesc_sw128(s0 + C::OFF_V, 16, 1024);  // V as K-major A
      const uint64_t dKt0 = sdesc_sw128(s0 + C::OFF_K, C::KBOX, 1024);            // K^T dims 0-127, MN-major A
      const uint64_t dKt1 = sdesc_sw128(s0 + C::OFF_K + C::KBOX, C::KBOX, 1024);  // K^T dims 64-191
      const uint64_t dS_mn = sdesc_sw128(s0 + C::OFF_DS, C::KBOX, 1024);          // dS^T as MN-major B
      auto kstep_a = [](int kk) { return (uint64_t)((((kk >> 2) * C::KBOX) + (kk & 3) * 32) >> 4); };
      auto kstep_b = [](int kk) { return (uint64_t)((((kk >> 2) * C::QBOX) + (kk & 3) * 32) >> 4); };
      auto issue_s = [&](int st) {
        const uint64_t bq = sdesc_sw128(s0 + C::OFF_Q + st * C::Q_BYTES, 16, 1024);
#pragma unroll
        for (int kk = 0; kk < kDqk / 16; ++kk)
          mma_ss(tmem + C::T_S, dK_k + kstep_a(kk), bq + kstep_b(kk), IDESC_S, kk > 0 ? 1u : 0u);
        mma_commit(&bar.s_full);
      };
      auto issue_dp = [&](int st) {
        const uint64_t bo = sdesc_sw128(s0 + C::OFF_DO + st * C::DO_BYTES, 16, 1024);
#pragma unroll
        for (int kk = 0; kk < kDv / 16; ++kk)
          mma_ss(tmem + C::T_DP, dV_k + kstep_a(kk), bo + kstep_b(kk), IDESC_S, kk > 0 ? 1u : 0u);
        mma_commit(&bar.dp_full);
      };
      auto issue_dv = [&](int st, bool acc) {
        const uint64_t bo = sdesc_sw128(s0 + C::OFF_DO + st * C::DO_BYTES, C::QBOX, 1024);
#pragma unroll
        for (int kk = 0; kk < kHalf / 16; ++kk)
          mma_ts(tmem + C::T_DV, tmem + C::T_S + packed_col<32>(kk * 16), bo + ((kk * 16 * 128) >> 4), IDESC_DV,
                 (acc || kk > 0) ? 1u : 0u);
      };
      auto issue_dk = [&](int st, bool acc) {
        const uint64_t bq = sdesc_sw128(s0 + C::OFF_Q + st * C::Q_BYTES, C::QBOX, 1024);
#pragma unroll
        for (int kk = 0; kk < kHalf / 16; ++kk)
          mma_ts(tmem + C::T_DK, tmem + C::T_DP + packed_col<32>(kk * 16), bq + ((kk * 16 * 128) >> 4), IDESC_DK,
                 (acc || kk > 0) ? 1u : 0u);
      };
      auto issue_dq = [&]() {
#pragma unroll
        for (int kk = 0; kk < kKeys / 16; ++kk)
          mma_ss(tmem + C::T_DP, dKt0 + ((kk * 16 * 128) >> 4), dS_mn + ((kk * 16 * 128) >> 4), IDESC_DQ,
                 kk > 0 ? 1u : 0u);
#pragma unroll
        for (int kk = 0; kk < kKeys / 16; ++kk)
          mma_ss(tmem + C::T_DQ1, dKt1 + ((kk * 16 * 128) >> 4), dS_mn + ((kk * 16 * 128) >> 4), IDESC_DQ,
                 kk > 0 ? 1u : 0u);
        mma_commit(&bar.ds_free);  // dQ^T was the dS^T tile's last reader
        mma_commit(&bar.dq_full);
      };

      int gs = 0;
      bool ok = true;
      for (int r = 0, uc = 0; ok; ++r) {
        const int ui = unit_index(a.cta_off, r, cta);
        if (ui < 0) break;
        const BwdUnit u = a.units[ui];
        int kmin, kmax;
        pm.range(u.t * kKeys, u.t * kKeys + kKeys, kmin, kmax);
        MStepIter<NAT> it;
        it.init(pm, u.h * G, u.h * G + G, kmin);
        if (!it.begin(pm)) continue;
        if (!(ok = mbar_wait(&bar.kv_full, uc & 1, ab))) break;
        tc_fence_after();
        // prologue: S and dP of the unit's first half-step
        if (!(ok = mbar_wait(&bar.q_full[gs & 1], (gs >> 1) & 1, ab))) break;
        tc_fence_after();
        bool more = !info[gs & 1].last;
        issue_s(gs & 1);
        if (gs > 0 && !(ok = mbar_wait(&bar.dq_free, (gs - 1) & 1, ab))) break;  // dQ of the last half-step read out
        if (!(ok = mbar_wait(&bar.do_full[gs & 1], (gs >> 1) & 1, ab))) break;
        tc_fence_after();
        issue_dp(gs & 1);
        for (int j = 0; ok; ++j, ++gs) {
          const int st = gs & 1;
          const bool this_more = more;
          if (!(ok = mbar_wait(&bar.p_full, gs & 1, ab))) break;
          tc_fence_after();
          issue_dv(st, j > 0);
          mma_commit(&bar.do_empty[st]);  // dO_j (dP_j, dV_j) is done
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
          if (gs > 0 && !(ok = mbar_wait(&bar.dq1_free, (gs - 1) & 1, ab))) break;  // the last dQ's second block read out
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
    // adds each staged dQ half-tile (six boxes of 32 columns x 64 rows) into
    // the fp32 accumulator, in slot order
    if (lane == 0) {
      int gs = 0;
      for (int r = 0;; ++r) {
        const int ui = unit_index(a.cta_off, r, cta);
        if (ui < 0) break;
        const BwdUnit u = a.units[ui];
        int kmin, kmax;
        pm.range(u.t * kKeys, u.t * kKeys + kKeys, kmin, kmax);
        MStepIter<NAT> it;
        it.init(pm, u.h * G, u.h * G + G, kmin);
        if (!it.begin(pm)) continue;
        do {
          const int hq = it.hq, qt = it.qt;
          for (int half = 0; half < 2; ++half) {
            // runs on after an abort: the staging is garbage, the waits bounded
            mbar_wait(&bar.staged, gs & 1, ab);
#pragma unroll
            for (int box = 0; box < 6; ++box)
              tma_reduce_add_4d(smem + C::OFF_STG + box * C::STG_BOX, &a.tdq, box * 32, hq, qt * kKeys + half * kHalf,
                                u.b);
            bulk_commit_group();
            mla_bulk_wait_read<0>();
            mbar_arrive(&bar.stg_free);  // the staging may be rewritten
            ++gs;
          }
        } while (it.next(pm));
      }
      bulk_wait_all();  // every dQ reduce has landed before the CTA retires
    }
  } else if (warp >= 12) {
    // ------------------------------------------------------------ dQ read-out
    // thread = TMEM lane = dim: dims 0-127 from dP's columns, dims 128-191
    // from lanes 64-127 of the second block; each thread writes its dims'
    // column of the staging boxes (query rows of 32 fp32, 128-byte swizzle)
    const int qd = warp & 3;
    const int lrow = (qd << 5) + lane;
    const uint32_t lane_base = uint32_t(qd * 32) << 16;
    auto stage_col = [&](int d, const uint32_t (&o)[32], int q0) {
      unsigned char* bx = smem + C::OFF_STG + (d >> 5) * C::STG_BOX;
      const int cc = d & 31;
#pragma unroll
      for (int q = 0; q < 32; ++q) {
        const int row = q0 + q;
        *reinterpret_cast<uint32_t*>(bx + row * 128 + ((((cc >> 2) ^ (row & 7))) << 4) + (cc & 3) * 4) = o[q];
      }
    };
    int gs = 0;
    for (int r = 0;; ++r) {
      const int ui = unit_index(a.cta_off, r, cta);
      if (ui < 0) break;
      const BwdUnit u = a.units[ui];
      int kmin, kmax;
      pm.range(u.t * kKeys, u.t * kKeys + kKeys, kmin, kmax);
      MStepIter<NAT> it;
      it.init(pm, u.h * G, u.h * G + G, kmin);
      if (!it.begin(pm)) continue;
      do {
        for (int half = 0; half < 2; ++half) {
          mbar_wait(&bar.dq_full, gs & 1, ab);  // runs on after an abort: the staging is garbage, the waits bounded
          tc_fence_after();
          uint32_t o0[32], o1[32];
          tmem_ld32(tmem + lane_base + C::T_DP, o0);
          tmem_ld32(tmem + lane_base + C::T_DP + 32, o1);
          tmem_ld_wait();
          tc_fence_before();
          mbar_arrive(&bar.dq_free);  // dP's columns: the next dP may go
          if (gs > 0) mbar_wait(&bar.stg_free, (gs - 1) & 1, ab);  // the last half-tile has left the staging
          stage_col(lrow, o0, 0);
          stage_col(lrow, o1, 32);
          tmem_ld32(tmem + lane_base + C::T_DQ1, o0);
          tmem_ld32(tmem + lane_base + C::T_DQ1 + 32, o1);
          tmem_ld_wait();
          tc_fence_before();
          mbar_arrive(&bar.dq1_free);  // the second block: the next dQ may go
          if (lrow >= 64) {  // lanes 64-127 of the second block hold dims 128-191
            stage_col(lrow + 64, o0, 0);
            stage_col(lrow + 64, o1, 32);
          }
          fence_proxy_async_smem();
          mbar_arrive(&bar.staged);
          ++gs;
        }
      } while (it.next(pm));
    }
  } else if (warp < 8) {
    // ------------------------------------------------------------ element-wise warps
    // Group g (warps 4g..4g+3) owns query columns [32g, 32g+32) of each
    // half-step's S^T/dP^T (thread = key row = TMEM lane) and, at the end of
    // a unit, dV columns [64g, 64g+64) and dK columns [96g, 96g+96).  A failed
    // wait (abort or timeout) runs on with whatever is in TMEM, so every role
    // walks all of its steps and every wait stays bounded.
    const int g = warp >> 2;
    const int row = ((warp & 3) << 5) + lane;  // TMEM lane
    const uint32_t lane_base = uint32_t((warp & 3) * 32) << 16;
    const uint64_t sl2x2 = f2pack(a.scale_log2, a.scale_log2);
    int gs = 0;

    for (int r = 0, uc = 0;; ++r) {
      const int ui = unit_index(a.cta_off, r, cta);
      if (ui < 0) break;
      const BwdUnit u = a.units[ui];
      const int kslot = u.t * kKeys + row;
      const bool kvalid = kslot < pm.S;
      const int kpos = kvalid ? pm.pos(kslot) : 0x7fffffff;
      int kmin, kmax;
      pm.range(u.t * kKeys, u.t * kKeys + kKeys, kmin, kmax);
      const bool k_inside = u.t * kKeys + kKeys <= pm.S;
      {
        MStepIter<NAT> it;
        it.init(pm, u.h * G, u.h * G + G, kmin);
        if (!it.begin(pm)) continue;
      }
      bool last;
      do {
        const int st = gs & 1;
        // ---- P into TMEM as bf16 (fp32 copy kept for dS)
        mbar_wait(&bar.s_full, gs & 1, ab);
        mbar_wait(&bar.q_full[st], (gs >> 1) & 1, ab);
        tc_fence_after();
        const int qt = info[st].qt, half = info[st].half;
        last = info[st].last != 0;
        const int slot0 = qt * kKeys + half * kHalf;
        const int qmin = info[st].qmin;  // (from the producer: no division on this path)
        const float* lse_s = reinterpret_cast<const float*>(smem + C::OFF_VEC + st * C::VEC_BYTES) + g * 32;
        const float* del_s = lse_s + kHalf;
        float p[32];
        const uint32_t t_s = tmem + lane_base + C::T_S + g * 32;
        const uint32_t t_pk = tmem + lane_base + C::T_S + packed_col<32>(g * 32);
        if ((kmax <= qmin) && k_inside && slot0 + kHalf <= pm.S)
          mla_ew_p<false>(t_s, t_pk, lse_s, sl2x2, p, kpos, pm, 0);
        else
          mla_ew_p<true>(t_s, t_pk, lse_s, sl2x2, p, kpos, pm, slot0 + g * 32);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&bar.p_full);
        // ---- dS = P * (dP - D): bf16 into TMEM (for dK), then shared memory (for dQ)
        mbar_wait(&bar.dp_full, gs & 1, ab);
        tc_fence_after();
        uint32_t dp[32], dk[16];
        tmem_ld32(tmem + lane_base + C::T_DP + g * 32, dp);
        tmem_ld_wait();
        const uint64_t* nd2 = reinterpret_cast<const uint64_t*>(del_s);
#pragma unroll
        for (int c = 0; c < 32; c += 2) {
          float d0, d1;
          f2unpack(f2mul(f2pack(p[c], p[c + 1]), f2add(f2pack_u(dp[c], dp[c + 1]), nd2[c >> 1])), d0, d1);
          dk[c >> 1] = pack_bf16(d0, d1);
        }
        tmem_st16(tmem + lane_base + C::T_DP + packed_col<32>(g * 32), dk);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&bar.dst_full);
        if (gs > 0) mbar_wait(&bar.ds_free, (gs - 1) & 1, ab);  // the last dQ^T has read the dS^T tile
        unsigned char* dsr = smem + C::OFF_DS + row * 128;  // this key row: 64 queries, 8 per 16-byte chunk
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int chunk = 4 * g + q;
          *reinterpret_cast<uint4*>(dsr + ((chunk ^ (row & 7)) << 4)) =
              make_uint4(dk[4 * q], dk[4 * q + 1], dk[4 * q + 2], dk[4 * q + 3]);
        }
        fence_proxy_async_smem();
        mbar_arrive(&bar.dss_full);
        ++gs;
      } while (!last);
      // dV and scale*dK of this key tile
      mbar_wait(&bar.acc_full, uc & 1, ab);
      tc_fence_after();
      const size_t krow = (size_t)u.b * pm.S + (kvalid ? mla_mem_row<NAT>(pm, kslot) : 0);
      const float sc = a.scale;
      // shared rope keys: dk holds the 128 nope columns per head, and the rope
      // columns are summed over heads into dk_rope_acc
      const bool rope = a.rope_shared != 0;
      __nv_bfloat16* dvp = static_cast<__nv_bfloat16*>(a.dv) + (krow * a.sh.Hkv + u.h) * kDv;
      __nv_bfloat16* dkp = static_cast<__nv_bfloat16*>(a.dk) + (krow * a.sh.Hkv + u.h) * (rope ? 128 : kDqk);
#pragma unroll 1
      for (int c0 = g * 64; c0 < g * 64 + 64; c0 += 32) {
        uint32_t o[32];
        tmem_ld32(tmem + lane_base + C::T_DV + c0, o);
        tmem_ld_wait();
        if (kvalid) {
          uint4* dst = reinterpret_cast<uint4*>(dvp + c0);
#pragma unroll
          for (int v4 = 0; v4 < 4; ++v4)
            dst[v4] = make_uint4(pack_bf16(__uint_as_float(o[8 * v4 + 0]), __uint_as_float(o[8 * v4 + 1])),
                                 pack_bf16(__uint_as_float(o[8 * v4 + 2]), __uint_as_float(o[8 * v4 + 3])),
                                 pack_bf16(__uint_as_float(o[8 * v4 + 4]), __uint_as_float(o[8 * v4 + 5])),
                                 pack_bf16(__uint_as_float(o[8 * v4 + 6]), __uint_as_float(o[8 * v4 + 7])));
        }
      }
#pragma unroll 1
      for (int c0 = g * 96; c0 < g * 96 + 96; c0 += 32) {
        uint32_t o[32];
        tmem_ld32(tmem + lane_base + C::T_DK + c0, o);
        tmem_ld_wait();
        if (kvalid && rope && c0 >= 128) {
          float* acc = a.dk_rope_acc + krow * 64 + (c0 - 128);
#pragma unroll
          for (int v4 = 0; v4 < 8; ++v4)
            mla_red_add_v4(acc + 4 * v4, sc * __uint_as_float(o[4 * v4 + 0]), sc * __uint_as_float(o[4 * v4 + 1]),
                       sc * __uint_as_float(o[4 * v4 + 2]), sc * __uint_as_float(o[4 * v4 + 3]));
        } else if (kvalid) {
          uint4* dst = reinterpret_cast<uint4*>(dkp + c0);
#pragma unroll
          for (int v4 = 0; v4 < 4; ++v4)
            dst[v4] = make_uint4(pack_bf16(sc * __uint_as_float(o[8 * v4 + 0]), sc * __uint_as_float(o[8 * v4 + 1])),
                                 pack_bf16(sc * __uint_as_float(o[8 * v4 + 2]), sc * __uint_as_float(o[8 * v4 + 3])),
                                 pack_bf16(sc * __uint_as_float(o[8 * v4 + 4]), sc * __uint_as_float(o[8 * v4 + 5])),
                                 pack_bf16(sc * __uint_as_float(o[8 * v4 + 6]), sc * __uint_as_float(o[8 * v4 + 7])));
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

template <bool NAT>
cudaError_t launch_mla(const BwdArgs& a, int grid, cudaStream_t st) {
  auto kern = attn_bwd_mla_kernel<NAT>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, MCfg::SMEM);
  if (e != cudaSuccess) return e;
  kern<<<grid, kThreadsM, MCfg::SMEM, st>>>(a);
  e = cudaGetLastError();
  if (e != cudaSuccess) {
    cudaFuncAttributes fa{};
    cudaFuncGetAttributes(&fa, kern);
    fprintf(stderr, "attn_bwd_mla: %s (regs %d, max threads %d, smem %d)\n", cudaGetErrorString(e), fa.numRegs,
            fa.maxThreadsPerBlock, MCfg::SMEM);
  }
  return e;
}

}  // namespace

cudaError_t launch_attn_bwd_mla(const BwdArgs& a, int grid, cudaStream_t st) {
  return PosMap::make(a.sh.S, a.sh.cp, a.sh.lb).lb == 2 ? launch_mla<true>(a, grid, st) : launch_mla<false>(a, grid, st);
}

}  // namespace cpattn
