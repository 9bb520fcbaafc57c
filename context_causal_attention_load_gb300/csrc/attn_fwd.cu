// Flash forward of load-balanced context-parallel causal attention on
// tcgen05 tensor cores.
//
// What it computes ("Add context parallelism", MaxText pull request 1445,
// Description): every cp shard's queries attend to the whole gathered K/V;
// tokens and the causal mask are reordered so that slot i sees slot j iff
// pos(j) <= pos(i).  All shards run in one persistent launch as independent
// work units.  MHA and MLA head layouts ("Add support for EP to context
// parallelism in self-attention", Main code changes) and grouped KV heads.
//
// Work unit = two 128-row query tiles that read the same KV head (two heads
// of a GQA group on the same rows, or two neighbouring row tiles of one
// head).  Their KV tiles are the union of the tiles either one can see;
// tiles every row of a query tile can see need no mask, tiles no row can see
// are skipped (load balancing follows from the reorder: every shard visits
// the same number of tiles).  The host deals the units out to the CTAs,
// heaviest first, each to the least-loaded CTA; a CTA runs its own list.
//
// CTA = 12 warps, one CTA per SM (all 512 TMEM columns):
//   warps 0-3  softmax group 0 (query tile 0, one thread per row)
//   warps 4-7  softmax group 1 (query tile 1)
//   warp  8    TMA producer: Q tiles, then one ring stage per key step
//              (K of the unit's first tile alone, then V_j with K_{j+1})
//   warp  9    MMA issuer (one thread): S_t = Q_t K^T into TMEM, and
//              O_t += P_t V with P_t read straight from TMEM
//   warps 10-11 idle (they complete the third warpgroup)
// setmaxnreg moves registers from the producer/MMA warpgroup (120 each) to
// the softmax warpgroups (192 each), so a thread holds its row's 128
// scores in registers: one TMEM load wait per tile, then max, exp2 and the
// packed-bf16 P, with fp32 pair (f32x2) arithmetic.
// TMEM columns: [t*256, t*256+128) = S_t, overwritten in place by P_t as
// packed bf16 (64 columns); [t*256+128, t*256+128+Dv) = O_t.
// The MMA thread interleaves the groups (PV_0, QK_0', PV_1, QK_1'), so one
// group's softmax runs while the tensor core serves the other.  Online
// softmax in the log2 domain with a lazy rescale: O_t is rescaled in TMEM
// only when a row maximum grows by more than 8 (a factor 256).
#include "common.cuh"
#include "internal.h"

namespace cpattn {
namespace {

constexpr int BM = 128;  // query rows per tile
constexpr int BN = 128;  // key rows per tile
constexpr int kThreads = 384;
constexpr int kRegsLaunch = 168;  // 65536 / 384, rounded down to a multiple of 8
constexpr int kRegsSoftmax = 192;
constexpr int kRegsOther = 120;
static_assert(2 * 128 * kRegsSoftmax + 128 * kRegsOther <= kThreads * kRegsLaunch, "register split");

// Ring of NK stages: stage g holds K in slot g % NK and V in slot g % NV
// (NV < NK only where shared memory has no room for a second V slot; then a
// stage's V waits for the previous stage instead of the one NK back).
template <int DQK, int DV>
struct FwdCfg {
  static constexpr int NK = DQK == 192 ? 2 : (DQK == 64 ? 4 : 2);
  static constexpr int NV = DQK == 192 ? 1 : (DQK == 64 ? 4 : 2);
  static_assert(NV == NK || NV == 1, "stage ring");
  static constexpr int Q_BYTES = BM * DQK * 2;
  static constexpr int K_BYTES = BN * DQK * 2;
  static constexpr int V_BYTES = BN * DV * 2;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + 2 * Q_BYTES;
  static constexpr int OFF_V = OFF_K + NK * K_BYTES;
  static constexpr int OFF_BAR = OFF_V + NV * V_BYTES;
  static constexpr int OFF_POS = OFF_BAR + 256;      // int kpos[2 groups][128]
  static constexpr int OFF_MISC = OFF_POS + 2 * BN * 4;
  static constexpr int SMEM = OFF_MISC + 64 + 1024;  // + alignment slack
  static_assert(SMEM <= 232448, "shared memory budget");
};

struct Bars {
  uint64_t q_full, q_empty;
  uint64_t kv_full[4], kv_empty[4];  // per ring stage
  uint64_t s_full[2], p_full[2], o_full[2];
  uint64_t kpos[2];  // per softmax group: key-position table written
  uint64_t done;
};
static_assert(sizeof(Bars) <= 256, "barrier area");

__device__ __forceinline__ int kv_bound(const PosMap& pm, const FwdUnit& u) {
  int mn, mx, mx2 = -1;
  pm.range(u.t0 * BM, u.t0 * BM + BM, mn, mx);
  if (u.h1 >= 0) pm.range(u.t1 * BM, u.t1 * BM + BM, mn, mx2);
  return mx > mx2 ? mx : mx2;
}

template <int DQK, int DV>
__global__ void __launch_bounds__(kThreads, 1) attn_fwd_kernel(const __grid_constant__ FwdArgs a) {
  using C = FwdCfg<DQK, DV>;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Bars& bar = *reinterpret_cast<Bars*>(smem + C::OFF_BAR);
  int* kpos_s = reinterpret_cast<int*>(smem + C::OFF_POS);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 16);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const PosMap pm = PosMap::make(a.sh.S, a.sh.cp, a.sh.lb);
  const Abort ab{abort_flag, a.err, a.wait_limit};

  if (tid == 0) {
    mbar_init(&bar.q_full, 1);
    mbar_init(&bar.q_empty, 1);
    for (int i = 0; i < C::NK; ++i) { mbar_init(&bar.kv_full[i], 1); mbar_init(&bar.kv_empty[i], 1); }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&bar.s_full[t], 1);
      mbar_init(&bar.p_full[t], 128);
      mbar_init(&bar.o_full[t], 1);
      mbar_init(&bar.kpos[t], 128);
    }
    mbar_init(&bar.done, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 9) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  if (warp == 8 && (tid & 31) == 0) {
    prefetch_tmap(&a.tq);
    prefetch_tmap(&a.tk);
    prefetch_tmap(&a.tv);
    if (a.rope_shared) prefetch_tmap(&a.tkr);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int cta = blockIdx.x;
  // each role's code sits under its own setmaxnreg, so the compiler
  // allocates it against that role's register budget
  if (warp >= 8) {
  regs_dec<kRegsOther>();
  if (warp == 8) {
    // ------------------------------------------------------------ producer
    if ((tid & 31) == 0) {
      int qph = 0;
      int ng = 0, nq = 0;  // ring stages and Q loads issued
      bool ok = true;
      // test hook (fault_skip_stage): one stage's loads are left out, so its
      // full barrier never completes and the MMA thread's bounded wait on it
      // runs out; everything after that is the ordinary abort path
      auto skipped = [&]() { return ng == a.fault_skip_stage; };
      // claim ring stage ng for `bytes` of loads (its K slot, and its V slot
      // when it carries V, must have been released)
      auto claim = [&](bool with_v, uint32_t bytes) {
        const int i = ng % C::NK;
        if (ng >= C::NK && !(ok = mbar_wait(&bar.kv_empty[i], ((ng / C::NK) & 1) ^ 1, ab))) return false;
        if (C::NV == 1 && with_v && ng >= 1) {
          const int pg = ng - 1;  // the stage before holds the one V slot
          if (!(ok = mbar_wait(&bar.kv_empty[pg % C::NK], (pg / C::NK) & 1, ab))) return false;
        }
        if (!skipped()) mbar_expect_tx(&bar.kv_full[i], bytes);
        return true;
      };
      auto load_k = [&](int kt, const FwdUnit& u) {
        if (skipped()) return;
        const int i = ng % C::NK;
        for (int bx = 0; bx < DQK / 64; ++bx) {
          unsigned char* dst = smem + C::OFF_K + i * C::K_BYTES + bx * BN * 128;
          if (DQK == 192 && bx == 2 && a.rope_shared)  // the shared rope keys
            tma_load_4d(dst, &a.tkr, &bar.kv_full[i], 0, 0, pm.row(kt * BN), u.b);
          else
            tma_load_4d(dst, &a.tk, &bar.kv_full[i], bx * 64, u.hkv, pm.row(kt * BN), u.b);
        }
      };
      auto load_v = [&](int kt, const FwdUnit& u) {
        if (skipped()) return;
        const int i = ng % C::NK, vi = ng % C::NV;
        for (int bx = 0; bx < DV / 64; ++bx)
          tma_load_4d(smem + C::OFF_V + vi * C::V_BYTES + bx * BN * 128, &a.tv, &bar.kv_full[i], bx * 64, u.hkv,
                      pm.row(kt * BN), u.b);
      };
      // while a unit's last stage is in flight, its successor's Q tiles and
      // first K/V tiles go to L2, so the loads at the unit boundary (which
      // wait for this unit's buffers) hit L2 instead of HBM
      auto prefetch_unit = [&](int r2) {
        const int ui2 = unit_index(a.cta_off, r2, cta);
        if (ui2 < 0) return;
        const FwdUnit u2 = a.units[ui2];
        const int kt0 = next_kv_tile(pm, BN, -1, kv_bound(pm, u2));
        for (int bx = 0; bx < DQK / 64; ++bx) {
          tma_prefetch_l2_4d(&a.tq, bx * 64, u2.h0, pm.row(u2.t0 * BM), u2.b);
          if (u2.h1 >= 0) tma_prefetch_l2_4d(&a.tq, bx * 64, u2.h1, pm.row(u2.t1 * BM), u2.b);
          if (kt0 >= 0) {
            if (DQK == 192 && bx == 2 && a.rope_shared)
              tma_prefetch_l2_4d(&a.tkr, 0, 0, pm.row(kt0 * BN), u2.b);
            else
              tma_prefetch_l2_4d(&a.tk, bx * 64, u2.hkv, pm.row(kt0 * BN), u2.b);
          }
        }
        for (int bx = 0; kt0 >= 0 && bx < DV / 64; ++bx) tma_prefetch_l2_4d(&a.tv, bx * 64, u2.hkv, pm.row(kt0 * BN), u2.b);
      };
      for (int r = 0; ok; ++r) {
        const int ui = unit_index(a.cta_off, r, cta);
        if (ui < 0) break;
        const FwdUnit u = a.units[ui];
        const bool has1 = u.h1 >= 0;
        if (r > 0) {
          if (!(ok = mbar_wait(&bar.q_empty, qph, ab))) break;
          qph ^= 1;
        }
        mbar_expect_tx(&bar.q_full, (has1 ? 2 : 1) * C::Q_BYTES);
        ++nq;
        for (int bx = 0; bx < DQK / 64; ++bx)
          tma_load_4d(smem + C::OFF_Q + bx * BM * 128, &a.tq, &bar.q_full, bx * 64, u.h0, pm.row(u.t0 * BM), u.b);
        if (has1)
          for (int bx = 0; bx < DQK / 64; ++bx)
            tma_load_4d(smem + C::OFF_Q + C::Q_BYTES + bx * BM * 128, &a.tq, &bar.q_full, bx * 64, u.h1,
                        pm.row(u.t1 * BM), u.b);
        KvWalk kw;
        kw.start(pm, BN, kv_bound(pm, u));
        int kt = kw.t;
        // prologue stage: the first K tile
        if (!claim(false, C::K_BYTES)) break;
        load_k(kt, u);
        ++ng;
        // step j: V_j and, unless it is the last, K_{j+1}
        while (kt >= 0) {
          kw.next(pm);
          const int nkt = kw.t;
          if (!claim(true, C::V_BYTES + (nkt >= 0 ? C::K_BYTES : 0))) break;
          load_v(kt, u);
          if (nkt >= 0) load_k(nkt, u);
          ++ng;
          if (nkt < 0) prefetch_unit(r + 1);
          kt = nkt;
        }
      }
      if (!ok) {
        // let the copies already issued land before the CTA exits: each wait
        // bounded on its own (a stage that never completes does not cut the
        // others' waits short)
        auto drain = [&](uint64_t* b, uint32_t parity) {
          volatile int own = 0;
          mbar_wait(b, parity, Abort{&own, a.err, a.wait_limit});
        };
        // stage g's loads complete phase g / NK of its barrier
        for (int g = ng - 1; g >= 0 && g >= ng - C::NK; --g) drain(&bar.kv_full[g % C::NK], (g / C::NK) & 1);
        if (nq > 0) drain(&bar.q_full, (nq - 1) & 1);
      }
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    if ((tid & 31) == 0) {
      constexpr uint32_t IDESC_QK = idesc_bf16(BM, BN, 0, 0);
      constexpr uint32_t IDESC_PV = idesc_bf16(BM, DV, 0, 1);
      const uint32_t sQ = smem_u32(smem + C::OFF_Q);
      const uint32_t sK = smem_u32(smem + C::OFF_K);
      const uint32_t sV = smem_u32(smem + C::OFF_V);
      int qph = 0;
      int pph[2] = {0, 0};
      bool ok = true;

      // descriptors advance by adding byte offsets / 16 to the start-address field;
      // the issue loops are unrolled: the MMA queue is shallow, so every
      // instruction this thread spends between MMAs shows as tensor-pipe idle
      auto issue_qk = [&](int t, int kslot) {
        const uint32_t d = tmem + t * 256;
        const uint64_t ad0 = sdesc_sw128(sQ + t * C::Q_BYTES, 16, 1024);
        const uint64_t bd0 = sdesc_sw128(sK + kslot * C::K_BYTES, 16, 1024);
#pragma unroll
        for (int kk = 0; kk < DQK / 16; ++kk) {
          const uint32_t off = ((kk >> 2) * (BM * 128) + (kk & 3) * 32) >> 4;  // BM == BN
          mma_ss(d, ad0 + off, bd0 + off, IDESC_QK, kk > 0 ? 1u : 0u);
        }
      };
      auto issue_pv = [&](int t, int vslot, bool acc) {
        const uint32_t d = tmem + t * 256 + 128;
        const uint32_t p = tmem + t * 256;
        const uint64_t bd0 = sdesc_sw128(sV + vslot * C::V_BYTES, BN * 128, 1024);
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk)
          mma_ts(d, p + kk * 8, bd0 + ((kk * 16 * 128) >> 4), IDESC_PV, (acc || kk > 0) ? 1u : 0u);
      };

      int g = 0;  // ring stage
      for (int r = 0; ok; ++r) {
        const int ui = unit_index(a.cta_off, r, cta);
        if (ui < 0) break;
        const FwdUnit u = a.units[ui];
        const bool has1 = u.h1 >= 0;
        const int nt = has1 ? 2 : 1;
        if (!(ok = mbar_wait(&bar.q_full, qph, ab))) break;
        qph ^= 1;
        tc_fence_after();
        // prologue stage: S_0 and S_1 of the first key tile
        if (!(ok = mbar_wait(&bar.kv_full[g % C::NK], (g / C::NK) & 1, ab))) break;
        tc_fence_after();
        for (int t = 0; t < nt; ++t) {
          issue_qk(t, g % C::NK);
          mma_commit(&bar.s_full[t]);
        }
        mma_commit(&bar.kv_empty[g % C::NK]);
        ++g;
        for (int j = 0; ok; ++j, ++g) {
          const bool more = j + 1 < u.nkv;
          if (!more) mma_commit(&bar.q_empty);  // every QK of this unit is issued
          if (!(ok = mbar_wait(&bar.kv_full[g % C::NK], (g / C::NK) & 1, ab))) break;
          for (int t = 0; t < nt; ++t) {
            if (!(ok = mbar_wait(&bar.p_full[t], pph[t], ab))) break;
            pph[t] ^= 1;
            tc_fence_after();
            issue_pv(t, g % C::NV, j > 0);
            if (!more) {
              mma_commit(&bar.o_full[t]);
            } else {
              issue_qk(t, g % C::NK);
              mma_commit(&bar.s_full[t]);
            }
          }
          if (!ok) break;
          mma_commit(&bar.kv_empty[g % C::NK]);
          if (!more) {
            ++g;
            break;
          }
        }
      }
      // wait for every issued MMA before TMEM is released
      mma_drain(&bar.done, a.err, a.wait_limit);
    }
  }
  } else {
    regs_inc<kRegsSoftmax>();
    // ------------------------------------------------------------ softmax groups
    const int t = warp >> 2;          // group
    const int row = tid & 127;        // query row in tile == TMEM lane
    const uint32_t lane_base = uint32_t((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + t * 256 + lane_base;
    const uint32_t tO = tS + 128;
    const float sl2 = a.scale_log2;
    int sph = 0, oph = 0, kbph = 0;
    bool ok = true;
    __nv_bfloat16* outp = static_cast<__nv_bfloat16*>(a.out);

    for (int r = 0; ok; ++r) {
      const int ui = unit_index(a.cta_off, r, cta);
      if (ui < 0) break;
      const FwdUnit u = a.units[ui];
      if (t == 1 && u.h1 < 0) continue;
      const int h = t ? u.h1 : u.h0;
      const int qt = t ? u.t1 : u.t0;
      const int bound = kv_bound(pm, u);
      const int qslot = qt * BM + row;
      const bool qvalid = qslot < pm.S;
      const int qpos = qvalid ? pm.pos(qslot) : -1;
      int qmin, qmax;
      pm.range(qt * BM, qt * BM + BM, qmin, qmax);

      float m = -INFINITY, l = 0.f;
      int j = 0;
      // the key tiles and their positions walked incrementally: this
      // bookkeeping runs on the softmax thread between two steps, sharing
      // its issue slots with the other tile's softmax (a division per step
      // here cost about a third of a step)
      KvWalk kw;
      kw.start(pm, BN, bound);
      for (; kw.t >= 0; kw.next(pm), ++j) {
        const int kt = kw.t, kmin = kw.kmin, kmax = kw.kmax;
        const bool inside = kt * BN + BN <= pm.S;
        const int cls = (kmin > qmax) ? 0 : ((kmax <= qmin && inside) ? 2 : 1);  // 0 none, 1 partial, 2 all
        const int* kp = kpos_s + t * BN;
        if (cls == 1) {
          // table of the key tile's original positions, shared by the group
          // (the group syncs again once every thread has read it)
          const int ks = kt * BN + row;
          kpos_s[t * BN + row] = ks < pm.S ? pm.pos(ks) : 0x7fffffff;
          mbar_arrive(&bar.kpos[t]);
          ok = mbar_wait(&bar.kpos[t], kbph, ab);
          kbph ^= 1;
          if (!(ok = __all_sync(0xffffffffu, ok))) break;
        }
        ok = mbar_wait(&bar.s_full[t], sph, ab);
        if (!(ok = __all_sync(0xffffffffu, ok))) break;
        sph ^= 1;
        tc_fence_after();
        float rowsum = 0.f;
        // online-softmax bookkeeping shared by both paths: lazy rescale of O
        // (in TMEM) and l when the row maximum grows by more than 2^8
        auto update_max = [&](float mx) {
          const float m_new = fmaxf(m, mx * sl2);
          const bool need = (m == -INFINITY) ? (m_new != -INFINITY) : (m_new > m + 8.0f);
          if (__any_sync(0xffffffffu, need && j > 0)) {
            const float alpha = (need && m != -INFINITY) ? fast_exp2(m - m_new) : (need ? 0.f : 1.0f);
            const uint64_t a2 = f2pack(alpha, alpha);
#pragma unroll 1
            for (int c0 = 0; c0 < DV; c0 += 32) {
              uint32_t o[32];
              tmem_ld32(tO + c0, o);
              tmem_ld_wait();
#pragma unroll
              for (int i = 0; i < 32; i += 2) {
                float x0, x1;
                f2unpack(f2mul(f2pack_u(o[i], o[i + 1]), a2), x0, x1);
                o[i] = __float_as_uint(x0);
                o[i + 1] = __float_as_uint(x1);
              }
              tmem_st32(tO + c0, o);
            }
            tmem_st_wait();
          }
          if (need) {
            l = (m == -INFINITY) ? 0.f : l * fast_exp2(m - m_new);
            m = m_new;
          }
          return (m == -INFINITY) ? 0.f : m;
        };
        const uint64_t sl2x2 = f2pack(sl2, sl2);
        if (cls == 0) {
          uint32_t z[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) z[i] = 0u;
          tmem_st32(tS + 0, z);
          tmem_st32(tS + 32, z);
        } else if (cls == 1) {
          // diagonal / ragged tile: mask with the key-position table, two
          // passes over TMEM 32 columns at a time
          float mx = -INFINITY;
#pragma unroll 1
          for (int q4 = 0; q4 < 4; ++q4) {
            uint32_t sr[32];
            tmem_ld32(tS + q4 * 32, sr);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (kp[q4 * 32 + i] <= qpos) mx = fmaxf(mx, __uint_as_float(sr[i]));
          }
          const float mref = update_max(mx);
          const uint64_t negm2 = f2pack(-mref, -mref);
          uint64_t sum2 = f2pack(0.f, 0.f);
#pragma unroll 1
          for (int q4 = 0; q4 < 4; ++q4) {
            uint32_t sr[32];
            tmem_ld32(tS + q4 * 32, sr);
            tmem_ld_wait();
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              float x0, x1;
              f2unpack(f2fma(f2pack_u(sr[2 * i], sr[2 * i + 1]), sl2x2, negm2), x0, x1);
              x0 = kp[q4 * 32 + 2 * i] <= qpos ? fast_exp2(x0) : 0.f;
              x1 = kp[q4 * 32 + 2 * i + 1] <= qpos ? fast_exp2(x1) : 0.f;
              sum2 = f2add(sum2, f2pack(x0, x1));
              pk[i] = pack_bf16(x0, x1);
            }
            tmem_st16(tS + q4 * 16, pk);
          }
          float r0, r1;
          f2unpack(sum2, r0, r1);
          rowsum = r0 + r1;
          tmem_st_wait();
          mbar_arrive(&bar.kpos[t]);  // table read; it may be rewritten
          ok = mbar_wait(&bar.kpos[t], kbph, ab);
          kbph ^= 1;
          if (!(ok = __all_sync(0xffffffffu, ok))) break;
        } else {
          // every key visible: the row's 128 scores stay in registers
          uint32_t sr[4][32];
          tmem_ld32(tS + 0, sr[0]);
          tmem_ld32(tS + 32, sr[1]);
          tmem_ld32(tS + 64, sr[2]);
          tmem_ld32(tS + 96, sr[3]);
          tmem_ld_wait();
          float mx4[4];
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            float v = __uint_as_float(sr[q4][0]);
#pragma unroll
            for (int i = 1; i < 31; i += 2)
              v = fmax3(v, __uint_as_float(sr[q4][i]), __uint_as_float(sr[q4][i + 1]));
            mx4[q4] = fmaxf(v, __uint_as_float(sr[q4][31]));
          }
          const float mref = update_max(fmax3(fmaxf(mx4[0], mx4[1]), mx4[2], mx4[3]));
          const uint64_t negm2 = f2pack(-mref, -mref);
          uint64_t sum2 = f2pack(0.f, 0.f);
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              float x0, x1;
              f2unpack(f2fma(f2pack_u(sr[q4][2 * i], sr[q4][2 * i + 1]), sl2x2, negm2), x0, x1);
              x0 = fast_exp2(x0);
              x1 = fast_exp2(x1);
              sum2 = f2add(sum2, f2pack(x0, x1));
              pk[i] = pack_bf16(x0, x1);
            }
            tmem_st16(tS + q4 * 16, pk);
          }
          float r0, r1;
          f2unpack(sum2, r0, r1);
          rowsum = r0 + r1;
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&bar.p_full[t]);
        l += rowsum;
      }
      if (!ok) break;
      // epilogue: O / l -> bf16, lse
      ok = mbar_wait(&bar.o_full[t], oph, ab);
      if (!(ok = __all_sync(0xffffffffu, ok))) break;
      oph ^= 1;
      tc_fence_after();
      const float inv_l = l > 0.f ? 1.0f / l : 0.f;
      const int qrow = qvalid ? pm.row(qslot) : 0;  // memory row of this query
      __nv_bfloat16* orow = outp + (((size_t)u.b * pm.S + qrow) * a.sh.Hq + h) * DV;
      {
        uint32_t o[DV / 32][32];
#pragma unroll
        for (int c = 0; c < DV / 32; ++c) tmem_ld32(tO + c * 32, o[c]);
        tmem_ld_wait();
        const uint64_t il2 = f2pack(inv_l, inv_l);
#pragma unroll
        for (int c = 0; c < DV / 32; ++c) {
          uint32_t pkd[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            float x0, x1;
            f2unpack(f2mul(f2pack_u(o[c][2 * i], o[c][2 * i + 1]), il2), x0, x1);
            pkd[i] = pack_bf16(x0, x1);
          }
          if (qvalid) {
            uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
            for (int i = 0; i < 4; ++i) dst[i] = make_uint4(pkd[4 * i], pkd[4 * i + 1], pkd[4 * i + 2], pkd[4 * i + 3]);
          }
        }
      }
      if (qvalid) {
        const float lse = l > 0.f ? (m + __log2f(l)) * 0.6931471805599453f : -INFINITY;
        a.lse[((size_t)u.b * a.sh.Hq + h) * pm.S + qrow] = lse;
      }
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

template <int DQK, int DV>
cudaError_t launch_t(const FwdArgs& a, int grid, cudaStream_t st) {
  auto kern = attn_fwd_kernel<DQK, DV>;
  // setmaxnreg.inc only succeeds if the launch reserved kRegsLaunch per thread
  cudaFuncAttributes fa;
  cudaError_t e0 = cudaFuncGetAttributes(&fa, kern);
  if (e0 != cudaSuccess) return e0;
  if (fa.numRegs != kRegsLaunch) return cudaErrorInvalidConfiguration;
  // more than half of an SM's shared memory: one CTA per SM, so the CTA's
  // 512-column TMEM allocation never waits for a neighbour
  const int smem = FwdCfg<DQK, DV>::SMEM > 120 * 1024 ? FwdCfg<DQK, DV>::SMEM : 120 * 1024;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  kern<<<grid, kThreads, smem, st>>>(a);
  return cudaGetLastError();
}

}  // namespace

int attn_fwd_smem_bytes(int Dqk, int Dv) {
  if (Dqk == 64) return FwdCfg<64, 64>::SMEM;
  if (Dqk == 128) return FwdCfg<128, 128>::SMEM;
  return FwdCfg<192, 128>::SMEM;
}

cudaError_t launch_attn_fwd(const FwdArgs& a, int grid, cudaStream_t st) {
  if (a.sh.Dqk == 64 && a.sh.Dv == 64) return launch_t<64, 64>(a, grid, st);
  if (a.sh.Dqk == 128 && a.sh.Dv == 128) return launch_t<128, 128>(a, grid, st);
  if (a.sh.Dqk == 192 && a.sh.Dv == 128) return launch_t<192, 128>(a, grid, st);
  return cudaErrorInvalidValue;
}

}  // namespace cpattn
