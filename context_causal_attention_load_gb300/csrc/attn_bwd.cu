// Flash backward of load-balanced context-parallel causal attention on
// tcgen05 tensor cores.
//
// The pages train with context parallelism ("Add context parallelism",
// MaxText pull request 1445, Tests: training runs; "rename context to
// context_autoregressive", Tests: separate flash block sizes for the dq and
// dkv passes) but give no formula; this is the textbook gradient of
// out = softmax(scale q k^T + mask) v under the reordered causal mask
// (query slot i sees key slot j iff pos(j) <= pos(i)):
//   D = rowsum(dO * O),  P = exp(scale q k^T - lse),  dV = P^T dO,
//   dP = dO V^T,  dS = P * (dP - D),  dQ = scale dS K,  dK = scale dS^T Q.
// dK/dV of a KV head sum over the query heads of its group and over every
// shard (the transpose of the K/V all-gather).
//
// Three launches, none of them with atomics (results are deterministic):
//  * preprocess: D and lse*log2(e) per query row, padded to 128 rows;
//  * dK/dV kernel, key-stationary: a CTA owns a 128-row key tile of one KV
//    head and walks every (query head of the group, 64-row query tile) that
//    can see it.  S^T = K Q^T and dP^T = V dO^T land in TMEM (128 key lanes
//    x 64 query columns, double buffered so the tensor core computes step
//    i+1 while the element-wise warps turn step i into P^T and dS^T, which
//    are written back to TMEM as bf16 and feed dV += P^T dO and
//    dK += dS^T Q straight from TMEM;
//  * dQ kernel, query-stationary: a CTA owns a 128-row query tile of one
//    head and walks the 64-row key tiles it sees; S = Q K^T and dP = dO V^T
//    in TMEM, dS back to TMEM as bf16, dQ += dS K.
// Warp roles as in the forward: warps 0-7 element-wise (two groups, each
// half of the columns), warp 8 TMA producer, warp 9 MMA issuer.
#include "common.cuh"
#include "internal.h"

namespace cpattn {

// fire-and-forget fp32 add of four consecutive floats (16-byte aligned) in global memory
__device__ __forceinline__ void red_add_v4(float* p, float x, float y, float z, float w) {
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(x), "f"(y), "f"(z), "f"(w) : "memory");
}

namespace {

constexpr int kThreads = 320;
constexpr int TK = 128;  // key rows per dk/dv unit; query rows per dq unit

// next query tile of T slots (> cur) that sees keys at position bound and
// holds a slot in [lo, hi) (the query slots taking part: all of them, or one
// shard's); tiles come in increasing slot order
__device__ __forceinline__ int next_q_tile_in(const PosMap& pm, int T, int cur, int bound, int lo, int hi) {
  if (cur < 0) cur = lo / T - 1;  // no tile before the first one holding lo can qualify
  for (int qt = next_q_tile(pm, T, cur, bound); qt >= 0; qt = next_q_tile(pm, T, qt, bound)) {
    if (qt * T >= hi) return -1;
    if (qt * T + T > lo) return qt;
  }
  return -1;
}


// ============================================================================
// preprocess: -lse*log2(e) (-inf past S) and -rowsum(dO*O) (0 past S), stored
// negated so the element-wise warps apply them with one fused multiply-add;
// layout [B, Hq, Spad] in slot order.  LPR = Dv/8 lanes per (b, h, s) row, each with one
// 16-byte load of out and of dout; rows go in output order (s fastest), so
// the row statistics are written and lse read contiguously.  With dq_acc,
// also zeroes the row of the fused kernel's fp32 dQ accumulator.
// ============================================================================
template <int LPR, bool NAT>
__global__ void __launch_bounds__(256) bwd_preprocess_kernel(const __nv_bfloat16* __restrict__ out,
                                                             const __nv_bfloat16* __restrict__ dout,
                                                             const float* __restrict__ lse, float* lse_l2,
                                                             float* delta, float* dq_acc, AttnShape sh, int Spad) {
  const long long nrows = (long long)sh.B * sh.Hq * Spad;
  const PosMap pm = PosMap::make(sh.S, sh.cp, sh.lb);
  const int sub = threadIdx.x % LPR;
  const unsigned gmask = ((1u << LPR) - 1u) << ((threadIdx.x & 31) & ~(LPR - 1));  // this row's lanes
  const long long stride = (long long)gridDim.x * blockDim.x / LPR;
  for (long long r = ((long long)blockIdx.x * blockDim.x + threadIdx.x) / LPR; r < nrows; r += stride) {
    const int s = int(r % Spad);
    const long long bh = r / Spad;
    const int h = int(bh % sh.Hq);
    const int b = int(bh / sh.Hq);
    const bool valid = s < sh.S;
    const int mrow = (valid && NAT) ? pm.pos(s) : s;  // memory row of slot s (natural order under zero-copy)
    float acc = 0.f;
    if (valid) {
      const size_t row = ((size_t)b * sh.S + mrow) * sh.Hq + h;
      const uint4 a = __ldcs(reinterpret_cast<const uint4*>(out + row * sh.Dv) + sub);
      const uint4 g = __ldcs(reinterpret_cast<const uint4*>(dout + row * sh.Dv) + sub);
      acc = fmaf(bf16lo(a.x), bf16lo(g.x), fmaf(bf16hi(a.x), bf16hi(g.x), acc));
      acc = fmaf(bf16lo(a.y), bf16lo(g.y), fmaf(bf16hi(a.y), bf16hi(g.y), acc));
      acc = fmaf(bf16lo(a.z), bf16lo(g.z), fmaf(bf16hi(a.z), bf16hi(g.z), acc));
      acc = fmaf(bf16lo(a.w), bf16lo(g.w), fmaf(bf16hi(a.w), bf16hi(g.w), acc));
      if (dq_acc) {
        float4* z = reinterpret_cast<float4*>(dq_acc + row * sh.Dqk);
        for (int c = sub; c < sh.Dqk / 4; c += LPR) z[c] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
#pragma unroll
    for (int o = LPR / 2; o; o >>= 1) acc += __shfl_xor_sync(gmask, acc, o);
    if (sub == 0) {
      delta[r] = -acc;
      lse_l2[r] = valid ? -lse[bh * sh.S + mrow] * 1.4426950408889634f : -INFINITY;
    }
  }
}

// ============================================================================
// dK / dV
// ============================================================================
template <int DQK, int DV, int BQ_, int NBUF>
struct KvCfg {
  static constexpr int BQ = BQ_;
  static constexpr int NQ = BQ_ == 128 ? (DQK == 64 ? 4 : 2) : (DQK == 192 ? 3 : 4);  // query stages
  static constexpr int K_BYTES = TK * DQK * 2;
  static constexpr int V_BYTES = TK * DV * 2;
  static constexpr int QT_BYTES = BQ * DQK * 2;
  static constexpr int DO_BYTES = BQ * DV * 2;
  static constexpr int VEC_BYTES = BQ * 4;
  static constexpr int ST_Q = 0;
  static constexpr int ST_DO = QT_BYTES;
  static constexpr int ST_LSE = ST_DO + DO_BYTES;
  static constexpr int ST_DEL = ST_LSE + VEC_BYTES;
  static constexpr int ST_POS = ST_DEL + VEC_BYTES;
  static constexpr int STAGE = (ST_POS + VEC_BYTES + 1023) / 1024 * 1024;
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = K_BYTES;
  static constexpr int OFF_ST = OFF_V + V_BYTES;
  static constexpr int OFF_BAR = OFF_ST + NQ * STAGE;
  static constexpr int OFF_MISC = OFF_BAR + 256;
  static constexpr int SMEM = OFF_MISC + 64 + 1024;
  static_assert(SMEM <= 232448, "shared memory budget");
  // TMEM columns
  static constexpr int T_S = 0;                  // S^T / P^T, buffer b at b*BQ
  static constexpr int T_DP = NBUF * BQ;         // dP^T / dS^T
  static constexpr int T_DV = 2 * NBUF * BQ;
  static constexpr int T_DK = T_DV + DV;
  static_assert(T_DK + DQK <= 512, "TMEM budget");
};

struct KvBars {
  uint64_t kv_full, kv_empty;
  uint64_t q_full[4], q_empty[4];
  uint64_t sd_full[2], ew_full[2];
  uint64_t acc_full;
  uint64_t done;
};

template <int DQK, int DV, int BQ_, int NBUF>
__global__ void __launch_bounds__(kThreads, 1) attn_bwd_dkdv_kernel(const __grid_constant__ BwdArgs a) {
  using C = KvCfg<DQK, DV, BQ_, NBUF>;
  constexpr int BQ = C::BQ;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  KvBars& bar = *reinterpret_cast<KvBars*>(smem + C::OFF_BAR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 16);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const PosMap pm = PosMap::make(a.sh.S, a.sh.cp, a.sh.lb);
  const Abort ab{abort_flag, a.err};
  const int G = a.sh.Hq / a.sh.Hkv;

  if (tid == 0) {
    mbar_init(&bar.kv_full, 1);
    mbar_init(&bar.kv_empty, 1);
    for (int i = 0; i < C::NQ; ++i) { mbar_init(&bar.q_full[i], 1); mbar_init(&bar.q_empty[i], 1); }
    for (int i = 0; i < 2; ++i) { mbar_init(&bar.sd_full[i], 1); mbar_init(&bar.ew_full[i], 256); }
    mbar_init(&bar.acc_full, 1);
    mbar_init(&bar.done, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 9) { tmem_alloc(tmem_slot, 512); tmem_relinquish(); }
  if (warp == 8 && lane == 0) {
    prefetch_tmap(&a.tq); prefetch_tmap(&a.tk); prefetch_tmap(&a.tv); prefetch_tmap(&a.tdo);
    if (a.rope_shared) prefetch_tmap(&a.tkr);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int cta = blockIdx.x;

  if (warp == 8) {
    // ------------------------------------------------------------ producer (whole warp)
    int qs = 0, qph = 0, kvph = 0;
    bool ok = true;
    for (int r = 0; ok; ++r) {
      const int ui = unit_index(a.cta_off, r, cta);
      if (ui < 0) break;
      const BwdUnit u = a.units[ui];
      if (lane == 0) {
        ok = mbar_wait(&bar.kv_empty, kvph ^ 1, ab);
        if (ok) {
          mbar_expect_tx(&bar.kv_full, C::K_BYTES + C::V_BYTES);
          for (int bx = 0; bx < DQK / 64; ++bx) {
            if (DQK == 192 && bx == 2 && a.rope_shared)  // the shared rope keys
              tma_load_4d(smem + C::OFF_K + bx * TK * 128, &a.tkr, &bar.kv_full, 0, 0, pm.row(u.t * TK), u.b);
            else
              tma_load_4d(smem + C::OFF_K + bx * TK * 128, &a.tk, &bar.kv_full, bx * 64, u.h, pm.row(u.t * TK), u.b);
          }
          for (int bx = 0; bx < DV / 64; ++bx)
            tma_load_4d(smem + C::OFF_V + bx * TK * 128, &a.tv, &bar.kv_full, bx * 64, u.h, pm.row(u.t * TK), u.b);
        }
      }
      kvph ^= 1;
      if (!(ok = __shfl_sync(0xffffffffu, ok, 0))) break;
      int kmin, kmax;
      pm.range(u.t * TK, u.t * TK + TK, kmin, kmax);
      for (int hq = u.h * G; hq < u.h * G + G && ok; ++hq) {
        for (int qt = next_q_tile_in(pm, BQ, -1, kmin, a.q_lo, a.q_hi); qt >= 0;
             qt = next_q_tile_in(pm, BQ, qt, kmin, a.q_lo, a.q_hi)) {
          if (lane == 0) ok = mbar_wait(&bar.q_empty[qs], qph ^ 1, ab);
          if (!(ok = __shfl_sync(0xffffffffu, ok, 0))) break;
          unsigned char* st = smem + C::OFF_ST + qs * C::STAGE;
          int* qp = reinterpret_cast<int*>(st + C::ST_POS);
          for (int i = lane; i < BQ; i += 32) {  // rows outside the slots taking part see no key
            const int s = qt * BQ + i;
            qp[i] = (s < pm.S && s >= a.q_lo && s < a.q_hi) ? pm.pos(s) : -1;
          }
          __syncwarp();
          if (lane == 0) {
            mbar_expect_tx(&bar.q_full[qs], C::QT_BYTES + C::DO_BYTES + 2 * C::VEC_BYTES);
            for (int bx = 0; bx < DQK / 64; ++bx)
              tma_load_4d(st + C::ST_Q + bx * BQ * 128, &a.tq, &bar.q_full[qs], bx * 64, hq, pm.row(qt * BQ), u.b);
            for (int bx = 0; bx < DV / 64; ++bx)
              tma_load_4d(st + C::ST_DO + bx * BQ * 128, &a.tdo, &bar.q_full[qs], bx * 64, hq, pm.row(qt * BQ), u.b);
            const size_t vo = ((size_t)u.b * a.sh.Hq + hq) * a.Spad + (size_t)qt * BQ;
            bulk_load(st + C::ST_LSE, a.lse_l2 + vo, C::VEC_BYTES, &bar.q_full[qs]);
            bulk_load(st + C::ST_DEL, a.delta + vo, C::VEC_BYTES, &bar.q_full[qs]);
          }
          if (++qs == C::NQ) { qs = 0; qph ^= 1; }
        }
      }
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t IDESC_S = idesc_bf16(TK, BQ, 0, 0);   // S^T, dP^T: K-major x K-major
      constexpr uint32_t IDESC_DV = idesc_bf16(TK, DV, 0, 1);  // P^T(tmem) x dO (MN-major)
      constexpr uint32_t IDESC_DK = idesc_bf16(TK, DQK, 0, 1); // dS^T(tmem) x Q (MN-major)
      const uint32_t sK = smem_u32(smem + C::OFF_K);
      const uint32_t sV = smem_u32(smem + C::OFF_V);
      const uint32_t sSt = smem_u32(smem + C::OFF_ST);
      int qs = 0, qph = 0, kvph = 0;
      int ewph[2] = {0, 0};
      bool ok = true;

      // descriptors: base computed once, k-steps add byte offsets / 16 to
      // the start-address field (keeps the single issuing thread fast)
      const uint64_t dK0 = sdesc_sw128(sK, 16, 1024), dV0 = sdesc_sw128(sV, 16, 1024);
      auto issue_sdp = [&](int buf, int stage) {
        const uint32_t st = sSt + stage * C::STAGE;
        const uint64_t dQ0 = sdesc_sw128(st + C::ST_Q, 16, 1024), dO0 = sdesc_sw128(st + C::ST_DO, 16, 1024);
#pragma unroll
        for (int kk = 0; kk < DQK / 16; ++kk)
          mma_ss(tmem + C::T_S + buf * BQ, dK0 + (((kk >> 2) * (TK * 128) + (kk & 3) * 32) >> 4),
                 dQ0 + (((kk >> 2) * (BQ * 128) + (kk & 3) * 32) >> 4), IDESC_S, kk > 0 ? 1u : 0u);
#pragma unroll
        for (int kk = 0; kk < DV / 16; ++kk)
          mma_ss(tmem + C::T_DP + buf * BQ, dV0 + (((kk >> 2) * (TK * 128) + (kk & 3) * 32) >> 4),
                 dO0 + (((kk >> 2) * (BQ * 128) + (kk & 3) * 32) >> 4), IDESC_S, kk > 0 ? 1u : 0u);
      };
      auto issue_acc = [&](int buf, int stage, bool acc) {
        const uint32_t st = sSt + stage * C::STAGE;
        const uint64_t bdo0 = sdesc_sw128(st + C::ST_DO, BQ * 128, 1024);
        const uint64_t bq0 = sdesc_sw128(st + C::ST_Q, BQ * 128, 1024);
        // dV chain, then dK chain (one accumulator at a time)
#pragma unroll
        for (int kk = 0; kk < BQ / 16; ++kk)
          mma_ts(tmem + C::T_DV, tmem + C::T_S + buf * BQ + packed_col<BQ / 2>(kk * 16), bdo0 + ((kk * 16 * 128) >> 4),
                 IDESC_DV, (acc || kk > 0) ? 1u : 0u);
#pragma unroll
        for (int kk = 0; kk < BQ / 16; ++kk)
          mma_ts(tmem + C::T_DK, tmem + C::T_DP + buf * BQ + packed_col<BQ / 2>(kk * 16), bq0 + ((kk * 16 * 128) >> 4),
                 IDESC_DK, (acc || kk > 0) ? 1u : 0u);
      };

      for (int r = 0; ok; ++r) {
        const int ui = unit_index(a.cta_off, r, cta);
        if (ui < 0) break;
        const BwdUnit u = a.units[ui];
        if (!(ok = mbar_wait(&bar.kv_full, kvph, ab))) break;
        kvph ^= 1;
        tc_fence_after();
        int kmin, kmax;
        pm.range(u.t * TK, u.t * TK + TK, kmin, kmax);
        // flatten (head, query tile) steps; step i uses buffer i % NBUF and ring stage
        int hq = u.h * G, qt = next_q_tile_in(pm, BQ, -1, kmin, a.q_lo, a.q_hi);
        auto advance = [&](int& h_, int& t_) {
          t_ = next_q_tile_in(pm, BQ, t_, kmin, a.q_lo, a.q_hi);
          if (t_ < 0 && ++h_ < u.h * G + G) t_ = next_q_tile_in(pm, BQ, -1, kmin, a.q_lo, a.q_hi);
        };
        int cur_stage = qs;
        if (!(ok = mbar_wait(&bar.q_full[qs], qph, ab))) break;
        tc_fence_after();
        issue_sdp(0, qs);
        mma_commit(&bar.sd_full[0]);
        if (++qs == C::NQ) { qs = 0; qph ^= 1; }
        for (int i = 0; ok; ++i) {
          int nh = hq, nt = qt;
          advance(nh, nt);
          const bool has_next = nh < u.h * G + G && nt >= 0;
          int next_stage = qs;
          if (NBUF == 2 && has_next) {
            if (!(ok = mbar_wait(&bar.q_full[qs], qph, ab))) break;
            tc_fence_after();
            issue_sdp((i + 1) & 1, qs);
            mma_commit(&bar.sd_full[(i + 1) & 1]);
            if (++qs == C::NQ) { qs = 0; qph ^= 1; }
          }
          const int buf = NBUF == 2 ? (i & 1) : 0;
          if (!(ok = mbar_wait(&bar.ew_full[buf], ewph[buf], ab))) break;
          ewph[buf] ^= 1;
          tc_fence_after();
          issue_acc(buf, cur_stage, i > 0);
          mma_commit(&bar.q_empty[cur_stage]);
          if (!has_next) break;
          if (NBUF == 1) {
            if (!(ok = mbar_wait(&bar.q_full[qs], qph, ab))) break;
            tc_fence_after();
            issue_sdp(0, qs);
            mma_commit(&bar.sd_full[0]);
            if (++qs == C::NQ) { qs = 0; qph ^= 1; }
          }
          cur_stage = next_stage;
          hq = nh;
          qt = nt;
        }
        if (!ok) break;
        mma_commit(&bar.acc_full);
        mma_commit(&bar.kv_empty);
      }
      mma_drain(&bar.done, a.err);
    }
  } else {
    // ------------------------------------------------------------ element-wise groups
    const int g = warp >> 2;              // column half
    const int row = tid & 127;            // key row == TMEM lane
    const uint32_t lane_base = uint32_t((warp & 3) * 32) << 16;
    constexpr int HC = BQ / 2;            // query columns per group
    const float sl2 = a.scale_log2;
    int qs = 0, qph = 0, acc_ph = 0;
    int sdph[2] = {0, 0};
    bool ok = true;
    for (int r = 0; ok; ++r) {
      const int ui = unit_index(a.cta_off, r, cta);
      if (ui < 0) break;
      const BwdUnit u = a.units[ui];
      const int kslot = u.t * TK + row;
      const bool kvalid = kslot < pm.S;
      const int kpos = kvalid ? pm.pos(kslot) : 0x7fffffff;
      int kmin, kmax;
      pm.range(u.t * TK, u.t * TK + TK, kmin, kmax);
      const bool k_inside = u.t * TK + TK <= pm.S;
      int i = 0;
      for (int hq = u.h * G; hq < u.h * G + G && ok; ++hq) {
        for (int qt = next_q_tile_in(pm, BQ, -1, kmin, a.q_lo, a.q_hi); qt >= 0;
             qt = next_q_tile_in(pm, BQ, qt, kmin, a.q_lo, a.q_hi), ++i) {
          const int buf = NBUF == 2 ? (i & 1) : 0;
          ok = mbar_wait(&bar.q_full[qs], qph, ab);
          if (ok) ok = mbar_wait(&bar.sd_full[buf], sdph[buf], ab);
          if (!(ok = __all_sync(0xffffffffu, ok))) break;
          sdph[buf] ^= 1;
          tc_fence_after();
          const unsigned char* st = smem + C::OFF_ST + qs * C::STAGE;
          int qmin, qmax;
          pm.range(qt * BQ, qt * BQ + BQ, qmin, qmax);
          const bool full = (kmax <= qmin) && k_inside && qt * BQ >= a.q_lo && qt * BQ + BQ <= a.q_hi;
          const uint64_t sl2x2 = f2pack(sl2, sl2);
#pragma unroll 1
          for (int c0 = g * HC; c0 < (g + 1) * HC; c0 += 32) {
            const float* lse_s = reinterpret_cast<const float*>(st + C::ST_LSE) + c0;
            const float* del_s = reinterpret_cast<const float*>(st + C::ST_DEL) + c0;
            const int* qp_s = reinterpret_cast<const int*>(st + C::ST_POS) + c0;
            uint32_t sv[32], dp[32];
            tmem_ld32(tmem + lane_base + C::T_S + buf * BQ + c0, sv);
            tmem_ld32(tmem + lane_base + C::T_DP + buf * BQ + c0, dp);
            tmem_ld_wait();
            uint32_t pk[16], dk[16];
            const uint64_t* nl2 = reinterpret_cast<const uint64_t*>(lse_s);  // -lse*log2e pairs
            const uint64_t* nd2 = reinterpret_cast<const uint64_t*>(del_s);  // -D pairs
#pragma unroll
            for (int c = 0; c < 32; c += 2) {
              float p0, p1;
              f2unpack(f2fma(f2pack_u(sv[c], sv[c + 1]), sl2x2, nl2[c >> 1]), p0, p1);
              p0 = fast_exp2(p0);
              p1 = fast_exp2(p1);
              if (!full) {
                p0 = (kpos <= qp_s[c]) ? p0 : 0.f;
                p1 = (kpos <= qp_s[c + 1]) ? p1 : 0.f;
              }
              const uint64_t p2 = f2pack(p0, p1);
              float d0, d1;
              f2unpack(f2mul(p2, f2add(f2pack_u(dp[c], dp[c + 1]), nd2[c >> 1])), d0, d1);
              pk[c >> 1] = pack_bf16(p0, p1);
              dk[c >> 1] = pack_bf16(d0, d1);
            }
            // packed bf16 pairs stay inside this group's own column range (they
            // overwrite S / dP columns this thread has already read)
            tmem_st16(tmem + lane_base + C::T_S + buf * BQ + packed_col<HC>(c0), pk);
            tmem_st16(tmem + lane_base + C::T_DP + buf * BQ + packed_col<HC>(c0), dk);
          }
          tmem_st_wait();
          tc_fence_before();
          mbar_arrive(&bar.ew_full[buf]);
          if (++qs == C::NQ) { qs = 0; qph ^= 1; }
        }
      }
      if (!ok) break;
      // epilogue: dV and scale*dK for this key tile, this group's column half
      ok = mbar_wait(&bar.acc_full, acc_ph, ab);
      if (!(ok = __all_sync(0xffffffffu, ok))) break;
      acc_ph ^= 1;
      tc_fence_after();
      const size_t krow = (size_t)u.b * pm.S + (kvalid ? pm.row(kslot) : 0);
      __nv_bfloat16* dvp = static_cast<__nv_bfloat16*>(a.dv) + (krow * a.sh.Hkv + u.h) * DV;
      // shared rope keys: dk holds the 128 nope columns per head, and the rope
      // columns are summed over heads into dk_rope_acc
      const bool rope = DQK == 192 && a.rope_shared;
      __nv_bfloat16* dkp = static_cast<__nv_bfloat16*>(a.dk) + (krow * a.sh.Hkv + u.h) * (rope ? 128 : DQK);
#pragma unroll 1
      for (int c0 = g * (DV / 2); c0 < (g + 1) * (DV / 2); c0 += 32) {
        uint32_t o[32];
        tmem_ld32(tmem + lane_base + C::T_DV + c0, o);
        tmem_ld_wait();
        if (kvalid && a.dv_part) {  // one shard's contribution, unrounded
          float4* dst = reinterpret_cast<float4*>(a.dv_part + (krow * a.sh.Hkv + u.h) * DV + c0);
#pragma unroll
          for (int v4 = 0; v4 < 8; ++v4)
            dst[v4] = make_float4(__uint_as_float(o[4 * v4 + 0]), __uint_as_float(o[4 * v4 + 1]),
                                  __uint_as_float(o[4 * v4 + 2]), __uint_as_float(o[4 * v4 + 3]));
        }
        if (kvalid && a.dv) {
          uint4* dst = reinterpret_cast<uint4*>(dvp + c0);
#pragma unroll
          for (int v4 = 0; v4 < 4; ++v4)
            dst[v4] = make_uint4(pack_bf16(__uint_as_float(o[8 * v4 + 0]), __uint_as_float(o[8 * v4 + 1])),
                                 pack_bf16(__uint_as_float(o[8 * v4 + 2]), __uint_as_float(o[8 * v4 + 3])),
                                 pack_bf16(__uint_as_float(o[8 * v4 + 4]), __uint_as_float(o[8 * v4 + 5])),
                                 pack_bf16(__uint_as_float(o[8 * v4 + 6]), __uint_as_float(o[8 * v4 + 7])));
        }
      }
      const float sc = a.scale;
#pragma unroll 1
      for (int c0 = g * (DQK / 2); c0 < (g + 1) * (DQK / 2); c0 += 32) {
        uint32_t o[32];
        tmem_ld32(tmem + lane_base + C::T_DK + c0, o);
        tmem_ld_wait();
        if (kvalid && a.dk_part) {  // one shard's contribution, unrounded (no shared rope key here)
          float4* dst = reinterpret_cast<float4*>(a.dk_part + (krow * a.sh.Hkv + u.h) * DQK + c0);
#pragma unroll
          for (int v4 = 0; v4 < 8; ++v4)
            dst[v4] = make_float4(sc * __uint_as_float(o[4 * v4 + 0]), sc * __uint_as_float(o[4 * v4 + 1]),
                                  sc * __uint_as_float(o[4 * v4 + 2]), sc * __uint_as_float(o[4 * v4 + 3]));
        }
        if (kvalid && rope && c0 >= 128) {
          float* acc = a.dk_rope_acc + krow * 64 + (c0 - 128);
#pragma unroll
          for (int v4 = 0; v4 < 8; ++v4)
            red_add_v4(acc + 4 * v4, sc * __uint_as_float(o[4 * v4 + 0]), sc * __uint_as_float(o[4 * v4 + 1]),
                       sc * __uint_as_float(o[4 * v4 + 2]), sc * __uint_as_float(o[4 * v4 + 3]));
        } else if (kvalid && a.dk) {
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

// ============================================================================
// dQ
// ============================================================================
template <int DQK, int DV, int BK_, int NSB_, int NDPB_>
struct QCfg {
  static constexpr int BK = BK_;      // key rows per step
  static constexpr int NSB = NSB_;    // S / dS TMEM buffers
  static constexpr int NDPB = NDPB_;  // dP TMEM buffers
  static constexpr int NS = BK_ == 128 ? 2 : (DQK == 192 ? 3 : 4);  // key/value stages
  static constexpr int Q_BYTES = TK * DQK * 2;
  static constexpr int DO_BYTES = TK * DV * 2;
  static constexpr int K_BYTES = BK * DQK * 2;
  static constexpr int V_BYTES = BK * DV * 2;
  static constexpr int ST_K = 0;
  static constexpr int ST_V = K_BYTES;
  static constexpr int ST_POS = ST_V + V_BYTES;
  static constexpr int STAGE = (ST_POS + BK * 4 + 1023) / 1024 * 1024;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_DO = Q_BYTES;
  static constexpr int OFF_ST = OFF_DO + DO_BYTES;
  static constexpr int OFF_BAR = OFF_ST + NS * STAGE;
  static constexpr int OFF_MISC = OFF_BAR + 256;
  static constexpr int SMEM = OFF_MISC + 64 + 1024;
  static_assert(SMEM <= 232448, "shared memory budget");
  static constexpr int T_S = 0;                 // S / dS (bf16), buffer b at b*BK
  static constexpr int T_DP = NSB * BK;         // dP, buffer b at T_DP + b*BK
  static constexpr int T_DQ = (NSB + NDPB) * BK;
  static_assert(T_DQ + DQK <= 512, "TMEM budget");
};

struct QBars {
  uint64_t q_full, q_empty;
  uint64_t kv_full[4], kv_empty[4];
  uint64_t sd_full[2], ew_full[2];
  uint64_t acc_full;
  uint64_t done;
};

template <int DQK, int DV, int BK_, int NSB, int NDPB>
__global__ void __launch_bounds__(kThreads, 1) attn_bwd_dq_kernel(const __grid_constant__ BwdArgs a) {
  using C = QCfg<DQK, DV, BK_, NSB, NDPB>;
  constexpr int BK = C::BK;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  QBars& bar = *reinterpret_cast<QBars*>(smem + C::OFF_BAR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 16);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const PosMap pm = PosMap::make(a.sh.S, a.sh.cp, a.sh.lb);
  const Abort ab{abort_flag, a.err};
  const int G = a.sh.Hq / a.sh.Hkv;

  if (tid == 0) {
    mbar_init(&bar.q_full, 1);
    mbar_init(&bar.q_empty, 1);
    for (int i = 0; i < C::NS; ++i) { mbar_init(&bar.kv_full[i], 1); mbar_init(&bar.kv_empty[i], 1); }
    for (int i = 0; i < 2; ++i) { mbar_init(&bar.sd_full[i], 1); mbar_init(&bar.ew_full[i], 256); }
    mbar_init(&bar.acc_full, 1);
    mbar_init(&bar.done, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 9) { tmem_alloc(tmem_slot, 512); tmem_relinquish(); }
  if (warp == 8 && lane == 0) {
    prefetch_tmap(&a.tq); prefetch_tmap(&a.tk); prefetch_tmap(&a.tv); prefetch_tmap(&a.tdo);
    if (a.rope_shared) prefetch_tmap(&a.tkr);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int cta = blockIdx.x;

  auto q_bound = [&](const BwdUnit& u) {
    int mn, mx;
    pm.range(u.t * TK, u.t * TK + TK, mn, mx);
    return mx;
  };

  if (warp == 8) {
    // ------------------------------------------------------------ producer (whole warp)
    int ks = 0, kph = 0, qph = 0;
    bool ok = true;
    for (int r = 0; ok; ++r) {
      const int ui = unit_index(a.cta_off, r, cta);
      if (ui < 0) break;
      const BwdUnit u = a.units[ui];
      const int hkv = u.h / G;
      if (lane == 0) {
        ok = mbar_wait(&bar.q_empty, qph ^ 1, ab);
        if (ok) {
          mbar_expect_tx(&bar.q_full, C::Q_BYTES + C::DO_BYTES);
          for (int bx = 0; bx < DQK / 64; ++bx)
            tma_load_4d(smem + C::OFF_Q + bx * TK * 128, &a.tq, &bar.q_full, bx * 64, u.h, pm.row(u.t * TK), u.b);
          for (int bx = 0; bx < DV / 64; ++bx)
            tma_load_4d(smem + C::OFF_DO + bx * TK * 128, &a.tdo, &bar.q_full, bx * 64, u.h, pm.row(u.t * TK), u.b);
        }
      }
      qph ^= 1;
      if (!(ok = __shfl_sync(0xffffffffu, ok, 0))) break;
      const int bound = q_bound(u);
      for (int kt = next_kv_tile(pm, BK, -1, bound); kt >= 0; kt = next_kv_tile(pm, BK, kt, bound)) {
        if (lane == 0) ok = mbar_wait(&bar.kv_empty[ks], kph ^ 1, ab);
        if (!(ok = __shfl_sync(0xffffffffu, ok, 0))) break;
        unsigned char* st = smem + C::OFF_ST + ks * C::STAGE;
        int* kp = reinterpret_cast<int*>(st + C::ST_POS);
        for (int i = lane; i < BK; i += 32) {
          const int s = kt * BK + i;
          kp[i] = s < pm.S ? pm.pos(s) : 0x7fffffff;
        }
        __syncwarp();
        if (lane == 0) {
          mbar_expect_tx(&bar.kv_full[ks], C::K_BYTES + C::V_BYTES);
          for (int bx = 0; bx < DQK / 64; ++bx) {
            if (DQK == 192 && bx == 2 && a.rope_shared)  // the shared rope keys
              tma_load_4d(st + C::ST_K + bx * BK * 128, &a.tkr, &bar.kv_full[ks], 0, 0, pm.row(kt * BK), u.b);
            else
              tma_load_4d(st + C::ST_K + bx * BK * 128, &a.tk, &bar.kv_full[ks], bx * 64, hkv, pm.row(kt * BK), u.b);
          }
          for (int bx = 0; bx < DV / 64; ++bx)
            tma_load_4d(st + C::ST_V + bx * BK * 128, &a.tv, &bar.kv_full[ks], bx * 64, hkv, pm.row(kt * BK), u.b);
        }
        if (++ks == C::NS) { ks = 0; kph ^= 1; }
      }
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t IDESC_S = idesc_bf16(TK, BK, 0, 0);
      constexpr uint32_t IDESC_DQ = idesc_bf16(TK, DQK, 0, 1);
      const uint32_t sQ = smem_u32(smem + C::OFF_Q);
      const uint32_t sDO = smem_u32(smem + C::OFF_DO);
      const uint32_t sSt = smem_u32(smem + C::OFF_ST);
      int ks = 0, kph = 0, qph = 0;
      int ewph[2] = {0, 0};
      bool ok = true;
      const uint64_t dQ0 = sdesc_sw128(sQ, 16, 1024), dO0 = sdesc_sw128(sDO, 16, 1024);
      auto issue_s = [&](int i, int stage) {  // S_i = Q K_i^T
        const uint64_t dK0 = sdesc_sw128(sSt + stage * C::STAGE + C::ST_K, 16, 1024);
#pragma unroll
        for (int kk = 0; kk < DQK / 16; ++kk)
          mma_ss(tmem + C::T_S + (i % NSB) * BK, dQ0 + (((kk >> 2) * (TK * 128) + (kk & 3) * 32) >> 4),
                 dK0 + (((kk >> 2) * (BK * 128) + (kk & 3) * 32) >> 4), IDESC_S, kk > 0 ? 1u : 0u);
      };
      auto issue_dp = [&](int i, int stage) {  // dP_i = dO V_i^T
        const uint64_t dV0 = sdesc_sw128(sSt + stage * C::STAGE + C::ST_V, 16, 1024);
#pragma unroll
        for (int kk = 0; kk < DV / 16; ++kk)
          mma_ss(tmem + C::T_DP + (i % NDPB) * BK, dO0 + (((kk >> 2) * (TK * 128) + (kk & 3) * 32) >> 4),
                 dV0 + (((kk >> 2) * (BK * 128) + (kk & 3) * 32) >> 4), IDESC_S, kk > 0 ? 1u : 0u);
      };
      auto issue_dq = [&](int i, int stage, bool acc) {  // dQ += dS_i K_i
        const uint64_t bd0 = sdesc_sw128(sSt + stage * C::STAGE + C::ST_K, BK * 128, 1024);
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk)
          mma_ts(tmem + C::T_DQ, tmem + C::T_S + (i % NSB) * BK + packed_col<BK / 2>(kk * 16), bd0 + ((kk * 16 * 128) >> 4),
                 IDESC_DQ, (acc || kk > 0) ? 1u : 0u);
      };
      for (int r = 0; ok; ++r) {
        const int ui = unit_index(a.cta_off, r, cta);
        if (ui < 0) break;
        const BwdUnit u = a.units[ui];
        const int bound = q_bound(u);
        if (!(ok = mbar_wait(&bar.q_full, qph, ab))) break;
        qph ^= 1;
        tc_fence_after();
        int kt = next_kv_tile(pm, BK, -1, bound);
        int cur_stage = ks;
        if (!(ok = mbar_wait(&bar.kv_full[ks], kph, ab))) break;
        tc_fence_after();
        issue_s(0, ks);
        issue_dp(0, ks);
        mma_commit(&bar.sd_full[0]);
        if (++ks == C::NS) { ks = 0; kph ^= 1; }
        // Step i: S_{i+1} / dP_{i+1} go ahead of dQ_i when they have a
        // buffer of their own (NSB / NDPB == 2); otherwise they follow dQ_i,
        // whose reads of dS_i they would overwrite (tcgen05 MMAs from one
        // thread execute in order).
        for (int i = 0; ok; ++i) {
          const int nkt = next_kv_tile(pm, BK, kt, bound);
          const int next_stage = ks;
          if (nkt >= 0) {
            if (!(ok = mbar_wait(&bar.kv_full[ks], kph, ab))) break;
            tc_fence_after();
            if (NSB == 2) issue_s(i + 1, ks);
            if (NDPB == 2) issue_dp(i + 1, ks);
            if (NSB == 2 && NDPB == 2) mma_commit(&bar.sd_full[(i + 1) & 1]);
          } else {
            mma_commit(&bar.q_empty);  // every S/dP MMA (the readers of Q and dO) is already issued
          }
          if (!(ok = mbar_wait(&bar.ew_full[i & 1], ewph[i & 1], ab))) break;
          ewph[i & 1] ^= 1;
          tc_fence_after();
          issue_dq(i, cur_stage, i > 0);
          mma_commit(&bar.kv_empty[cur_stage]);
          if (nkt < 0) break;
          if (NSB == 1) issue_s(i + 1, next_stage);
          if (NDPB == 1) issue_dp(i + 1, next_stage);
          if (NSB == 1 || NDPB == 1) mma_commit(&bar.sd_full[(i + 1) & 1]);
          if (++ks == C::NS) { ks = 0; kph ^= 1; }
          cur_stage = next_stage;
          kt = nkt;
        }
        if (!ok) break;
        mma_commit(&bar.acc_full);
      }
      mma_drain(&bar.done, a.err);
    }
  } else {
    // ------------------------------------------------------------ element-wise groups
    const int g = warp >> 2;
    const int row = tid & 127;  // query row == TMEM lane
    const uint32_t lane_base = uint32_t((warp & 3) * 32) << 16;
    constexpr int HC = BK / 2;  // key columns per group
    const float sl2 = a.scale_log2;
    int ks = 0, kph = 0, acc_ph = 0;
    int sdph[2] = {0, 0};
    bool ok = true;
    for (int r = 0; ok; ++r) {
      const int ui = unit_index(a.cta_off, r, cta);
      if (ui < 0) break;
      const BwdUnit u = a.units[ui];
      const int bound = q_bound(u);
      const int qslot = u.t * TK + row;
      const bool qvalid = qslot < pm.S;
      const int qpos = qvalid ? pm.pos(qslot) : -1;
      const size_t vo = ((size_t)u.b * a.sh.Hq + u.h) * a.Spad + qslot;
      const float nlse2 = a.lse_l2[vo];  // -lse*log2e
      const float ndel = a.delta[vo];    // -D
      int qmin, qmax;
      pm.range(u.t * TK, u.t * TK + TK, qmin, qmax);
      int i = 0;
      for (int kt = next_kv_tile(pm, BK, -1, bound); kt >= 0; kt = next_kv_tile(pm, BK, kt, bound), ++i) {
        const int buf = i & 1;
        ok = mbar_wait(&bar.kv_full[ks], kph, ab);
        if (ok) ok = mbar_wait(&bar.sd_full[buf], sdph[buf], ab);
        if (!(ok = __all_sync(0xffffffffu, ok))) break;
        sdph[buf] ^= 1;
        tc_fence_after();
        int kmin, kmax;
        pm.range(kt * BK, kt * BK + BK, kmin, kmax);
        const bool full = (kmax <= qmin) && (kt * BK + BK <= pm.S);
        const uint64_t sl2x2 = f2pack(sl2, sl2);
        const uint64_t nl2 = f2pack(nlse2, nlse2);
        const uint64_t nd2 = f2pack(ndel, ndel);
        const uint32_t tS = tmem + lane_base + C::T_S + (i % NSB) * BK;
        const uint32_t tP = tmem + lane_base + C::T_DP + (i % NDPB) * BK;
#pragma unroll 1
        for (int c0 = g * HC; c0 < (g + 1) * HC; c0 += 32) {
          const int* kp_s = reinterpret_cast<const int*>(smem + C::OFF_ST + ks * C::STAGE + C::ST_POS) + c0;
          uint32_t sv[32], dp[32];
          tmem_ld32(tS + c0, sv);
          tmem_ld32(tP + c0, dp);
          tmem_ld_wait();
          uint32_t dk[16];
#pragma unroll
          for (int c = 0; c < 32; c += 2) {
            float p0, p1;
            f2unpack(f2fma(f2pack_u(sv[c], sv[c + 1]), sl2x2, nl2), p0, p1);
            p0 = fast_exp2(p0);
            p1 = fast_exp2(p1);
            if (!full) {
              p0 = (kp_s[c] <= qpos) ? p0 : 0.f;
              p1 = (kp_s[c + 1] <= qpos) ? p1 : 0.f;
            }
            float d0, d1;
            f2unpack(f2mul(f2pack(p0, p1), f2add(f2pack_u(dp[c], dp[c + 1]), nd2)), d0, d1);
            dk[c >> 1] = pack_bf16(d0, d1);
          }
          // dS as packed bf16 inside this group's own column range
          tmem_st16(tS + packed_col<HC>(c0), dk);
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&bar.ew_full[buf]);
        if (++ks == C::NS) { ks = 0; kph ^= 1; }
      }
      if (!ok) break;
      ok = mbar_wait(&bar.acc_full, acc_ph, ab);
      if (!(ok = __all_sync(0xffffffffu, ok))) break;
      acc_ph ^= 1;
      tc_fence_after();
      __nv_bfloat16* dqp = static_cast<__nv_bfloat16*>(a.dq) + (((size_t)u.b * pm.S + (qvalid ? pm.row(qslot) : 0)) * a.sh.Hq + u.h) * DQK;
      const float sc = a.scale;
#pragma unroll 1
      for (int c0 = g * (DQK / 2); c0 < (g + 1) * (DQK / 2); c0 += 32) {
        uint32_t o[32];
        tmem_ld32(tmem + lane_base + C::T_DQ + c0, o);
        tmem_ld_wait();
        if (qvalid && qslot >= a.q_lo && qslot < a.q_hi) {  // one shard's rows only, for a shard
          uint4* dst = reinterpret_cast<uint4*>(dqp + c0);
#pragma unroll
          for (int v4 = 0; v4 < 4; ++v4)
            dst[v4] = make_uint4(pack_bf16(sc * __uint_as_float(o[8 * v4 + 0]), sc * __uint_as_float(o[8 * v4 + 1])),
                                 pack_bf16(sc * __uint_as_float(o[8 * v4 + 2]), sc * __uint_as_float(o[8 * v4 + 3])),
                                 pack_bf16(sc * __uint_as_float(o[8 * v4 + 4]), sc * __uint_as_float(o[8 * v4 + 5])),
                                 pack_bf16(sc * __uint_as_float(o[8 * v4 + 6]), sc * __uint_as_float(o[8 * v4 + 7])));
        }
      }
      tc_fence_before();
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

template <typename K>
cudaError_t launch_k(K kern, int smem, int grid, const BwdArgs& a, cudaStream_t st) {
  // more than half of an SM's shared memory: one CTA per SM, so the CTA's
  // 512-column TMEM allocation never waits for a neighbour
  if (smem < 120 * 1024) smem = 120 * 1024;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  kern<<<grid, kThreads, smem, st>>>(a);
  return cudaGetLastError();
}

}  // namespace

// Measured on GB300: 64-row steps with double-buffered S/dP (the element-wise
// work of one step overlaps the MMAs of the next, and four load stages keep
// the TMA copies off the critical path) beat 128-row steps, whose wider MMAs
// do not pay for the lost overlap and the shallower two-stage load ring.
int bwd_dkdv_q_tile(int) { return 64; }
int bwd_dq_kv_tile(int) { return 64; }

cudaError_t launch_bwd_preprocess(const void* out, const void* dout, const float* lse, float* lse_l2, float* delta,
                                  float* dq_acc, const AttnShape& sh, int Spad, cudaStream_t st) {
  const long long rows = (long long)sh.B * Spad * sh.Hq;
  const int lpr = sh.Dv / 8;  // Dv is 64 or 128
  long long blocks = (rows * lpr + 255) / 256;
  if (blocks > 152LL * 64) blocks = 152LL * 64;
  const bool nat = PosMap::make(sh.S, sh.cp, sh.lb).lb == 2;
  auto kern = lpr == 16 ? (nat ? bwd_preprocess_kernel<16, true> : bwd_preprocess_kernel<16, false>)
                        : (nat ? bwd_preprocess_kernel<8, true> : bwd_preprocess_kernel<8, false>);
  kern<<<(int)blocks, 256, 0, st>>>(static_cast<const __nv_bfloat16*>(out), static_cast<const __nv_bfloat16*>(dout),
                                    lse, lse_l2, delta, dq_acc, sh, Spad);
  return cudaGetLastError();
}

cudaError_t launch_attn_bwd_dkdv(const BwdArgs& a, int grid, cudaStream_t st) {
  if (a.sh.Dqk == 64) return launch_k(attn_bwd_dkdv_kernel<64, 64, 64, 2>, KvCfg<64, 64, 64, 2>::SMEM, grid, a, st);
  if (a.sh.Dqk == 128)
    return launch_k(attn_bwd_dkdv_kernel<128, 128, 64, 2>, KvCfg<128, 128, 64, 2>::SMEM, grid, a, st);
  // MLA: dK needs 192 TMEM columns, so S^T / dP^T are single-buffered
  return launch_k(attn_bwd_dkdv_kernel<192, 128, 64, 1>, KvCfg<192, 128, 64, 1>::SMEM, grid, a, st);
}

cudaError_t launch_attn_bwd_dq(const BwdArgs& a, int grid, cudaStream_t st) {
  if (a.sh.Dqk == 64) return launch_k(attn_bwd_dq_kernel<64, 64, 64, 2, 2>, QCfg<64, 64, 64, 2, 2>::SMEM, grid, a, st);
  if (a.sh.Dqk == 128)
    return launch_k(attn_bwd_dq_kernel<128, 128, 64, 2, 2>, QCfg<128, 128, 64, 2, 2>::SMEM, grid, a, st);
  return launch_k(attn_bwd_dq_kernel<192, 128, 64, 2, 2>, QCfg<192, 128, 64, 2, 2>::SMEM, grid, a, st);
}

}  // namespace cpattn
