// C ABI of libcpattn.so: argument checks, TMA descriptors, work lists,
// cached scratch, launches.  See include/cpattn.h for the contract.
#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <map>
#include <mutex>
#include <queue>
#include <string>
#include <tuple>
#include <vector>

#include "cpattn.h"
#include "common.cuh"
#include "internal.h"

using namespace cpattn;

namespace {

thread_local std::string g_last_error;

int fail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return code;
}

int cuda_fail(cudaError_t e, const char* what) {
  return fail(CPATTN_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

// ---- tensor maps -----------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

}  // namespace

// bf16 tensor map with 128-byte swizzle and zero fill past the extents
// (dims[0] innermost; strides in bytes for dims 1..rank-1)
int cpattn::encode_bf16_tmap(CUtensorMap* m, const void* ptr, int rank, const unsigned long long* dims,
                             const unsigned long long* strides, const unsigned* box) {
  return encode_tmap(m, ptr, rank, dims, strides, box, 2);
}

int cpattn::encode_tmap(CUtensorMap* m, const void* ptr, int rank, const unsigned long long* dims,
                        const unsigned long long* strides, const unsigned* box, int elem_bytes) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return -1;
  cuuint64_t d[5], st[4];
  cuuint32_t bx[5], es[5];
  for (int i = 0; i < rank; ++i) {
    d[i] = dims[i];
    bx[i] = box[i];
    es[i] = 1;
    if (i > 0) st[i - 1] = strides[i - 1];
  }
  const CUtensorMapDataType dt = elem_bytes == 1   ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                 : elem_bytes == 4 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                                   : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  CUresult r = fn(m, dt, rank,
                  const_cast<void*>(ptr), d, st, bx, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? 0 : -1;
}

namespace {

// [B, S, H, D] bf16 tensor seen as 4-D {D, H, S, B}; box = 64 columns x rows
// (128-byte rows, 128-byte swizzle, zero fill past S)
int make_tmap(CUtensorMap* m, const void* ptr, int B, int S, int H, int D, int rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return fail(CPATTN_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)S, (cuuint64_t)B};
  cuuint64_t strides[3] = {(cuuint64_t)D * 2, (cuuint64_t)H * D * 2, (cuuint64_t)S * H * D * 2};
  cuuint32_t box[4] = {64, 1, (cuuint32_t)rows, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(ptr), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(CPATTN_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  return CPATTN_OK;
}

// [B, S, H, D] fp32 tensor as 4-D {D, H, S, B}; box = 32 columns (128 bytes) x
// rows, 128-byte swizzle (the fused backward's dQ reduce-add target)
int make_tmap_f32(CUtensorMap* m, const void* ptr, int B, int S, int H, int D, int rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return fail(CPATTN_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)S, (cuuint64_t)B};
  cuuint64_t strides[3] = {(cuuint64_t)D * 4, (cuuint64_t)H * D * 4, (cuuint64_t)S * H * D * 4};
  cuuint32_t box[4] = {32, 1, (cuuint32_t)rows, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, const_cast<void*>(ptr), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(CPATTN_ERR_CUDA, "cuTensorMapEncodeTiled (fp32) failed (%d)", (int)r);
  return CPATTN_OK;
}

// ---- per-device state ---------------------------------------------------------
template <typename T>
struct DevBuf {
  T* ptr = nullptr;
  size_t n = 0;
};

// a work list dealt out to ncta CTAs: CTA c runs units [off[c], off[c+1])
template <typename U>
struct UnitPlan {
  DevBuf<U> units;
  DevBuf<int> off;
  int ncta = 0;
};

struct DevState {
  int num_sms = 0;
  int cc_major = 0, cc_minor = 0;
  int* err = nullptr;  // device error word
  std::map<std::vector<int>, UnitPlan<FwdUnit>> fwd_units;
  std::map<std::vector<int>, UnitPlan<BwdUnit>> bwd_units;
  DevBuf<float> bwd_stats;  // lse_l2 then delta
  DevBuf<float> dq_acc;     // fused backward's fp32 dQ accumulator
  DevBuf<float> rope_acc;   // MLA with shared rope keys: dK's rope columns summed over heads
  DevBuf<float> dec_o, dec_ml;
  DevBuf<float> mla_o, mla_ml;  // absorbed-MLA decode chunk partials
};

std::mutex g_mu;
std::map<int, DevState> g_dev;

// ---- optional per-launch timing (CUDA events on the launching stream) ------
struct ProfRec {
  const char* name;
  cudaEvent_t a, b;
};
bool g_prof_on = false;
std::vector<ProfRec> g_prof;
std::vector<cudaEvent_t> g_ev_pool;

cudaEvent_t prof_event() {
  if (!g_ev_pool.empty()) {
    cudaEvent_t e = g_ev_pool.back();
    g_ev_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  cudaEventCreate(&e);
  return e;
}

struct ProfScope {  // brackets one kernel launch when profiling is on
  cudaEvent_t b = nullptr;
  ProfScope(const char* name, cudaStream_t st) {
    if (!g_prof_on) return;
    ProfRec r{name, prof_event(), prof_event()};
    cudaEventRecord(r.a, st);
    b = r.b;
    g_prof.push_back(r);
    stream = st;
  }
  ~ProfScope() {
    if (b) cudaEventRecord(b, stream);
  }
  cudaStream_t stream = nullptr;
};

int get_state(DevState** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  DevState& s = g_dev[dev];
  if (!s.err) {
    cudaDeviceGetAttribute(&s.num_sms, cudaDevAttrMultiProcessorCount, dev);
    cudaDeviceGetAttribute(&s.cc_major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&s.cc_minor, cudaDevAttrComputeCapabilityMinor, dev);
    e = cudaMalloc(&s.err, sizeof(int));
    if (e != cudaSuccess) { s.err = nullptr; return fail(CPATTN_ERR_NO_MEMORY, "cudaMalloc(error word) failed"); }
    e = cudaMemset(s.err, 0, sizeof(int));
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemset");
  }
  *out = &s;
  return CPATTN_OK;
}

int need_sm103(const DevState& s) {
  if (s.cc_major != 10 || s.cc_minor != 3)
    return fail(CPATTN_ERR_UNSUPPORTED, "this library is built for sm_103a (GB300); device is sm_%d%d",
                s.cc_major, s.cc_minor);
  return CPATTN_OK;
}

template <typename T>
int ensure(DevBuf<T>& b, size_t n, cudaStream_t st, bool zero) {
  if (b.n >= n && b.ptr) return CPATTN_OK;
  if (b.ptr) {
    cudaStreamSynchronize(st);
    cudaFree(b.ptr);
    b.ptr = nullptr;
    b.n = 0;
  }
  cudaError_t e = cudaMalloc(&b.ptr, n * sizeof(T));
  if (e != cudaSuccess) {
    b.ptr = nullptr;
    return fail(CPATTN_ERR_NO_MEMORY, "cudaMalloc(%zu bytes) failed", n * sizeof(T));
  }
  if (zero) {
    e = cudaMemsetAsync(b.ptr, 0, n * sizeof(T), st);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync");
  }
  b.n = n;
  return CPATTN_OK;
}

template <typename T>
int upload(DevBuf<T>& b, const std::vector<T>& v) {
  cudaError_t e = cudaMalloc(&b.ptr, std::max<size_t>(1, v.size()) * sizeof(T));
  if (e != cudaSuccess) { b.ptr = nullptr; return fail(CPATTN_ERR_NO_MEMORY, "cudaMalloc(work list) failed"); }
  if (!v.empty()) {
    e = cudaMemcpy(b.ptr, v.data(), v.size() * sizeof(T), cudaMemcpyHostToDevice);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpy(work list)");
  }
  b.n = v.size();
  return CPATTN_OK;
}

// Deal a work list out to min(units, num_sms) CTAs so that the most loaded
// CTA carries as little as possible (every CTA then runs its units heaviest
// first).  The cost of a unit is its steps plus a fixed per-unit overhead
// measured in steps (pipeline fill and drain, epilogue), so many small units
// are not mistaken for little work.  With many units per CTA, units by
// decreasing cost each go to the least-loaded CTA (longest processing time
// first).  With few units per CTA that packs poorly (e.g. 3-4 units of
// similar cost per CTA), so the capacity of a CTA is searched instead: the
// smallest capacity for which first-fit-decreasing places every unit within
// the CTAs (MULTIFIT).  Its packing is kept only if it lowers the modelled
// maximum load by 3% or more: its CTAs are filled unevenly (the first ones
// tight with large units, the last ones with many small ones), which costs
// more than the model says (a full Llama2-shaped forward ran 6% slower under
// it for a modelled 1% gain).
template <typename U>
void plan_units(std::vector<std::pair<long long, U>> w, int num_sms, std::vector<U>& units,
                std::vector<int>& off, std::vector<long long>* cta_cost = nullptr) {
  std::stable_sort(w.begin(), w.end(), [](const auto& x, const auto& y) { return x.first > y.first; });
  const int ncta = (int)std::min<size_t>(w.size(), (size_t)std::max(1, num_sms));
  const size_t n = w.size();
  std::vector<int> bin(n, 0);  // CTA of each unit (in sorted order)
  long long best = 0;
  {
    using Load = std::pair<long long, int>;  // (cost so far, CTA): ties go to the lower CTA
    std::priority_queue<Load, std::vector<Load>, std::greater<Load>> pq;
    for (int c = 0; c < ncta; ++c) pq.push({0, c});
    for (size_t i = 0; i < n; ++i) {
      const Load top = pq.top();
      pq.pop();
      bin[i] = top.second;
      best = std::max(best, top.first + w[i].first);
      pq.push({top.first + w[i].first, top.second});
    }
  }
  if (n > 0 && n <= (size_t)ncta * 8) {
    long long total = 0;
    for (const auto& cu : w) total += cu.first;
    long long lo = std::max((total + ncta - 1) / ncta, n ? w[0].first : 0) - 1;  // infeasible
    long long hi = best;                                                        // feasible (LPT's load)
    std::vector<int> fit(n), fit_best;
    std::vector<long long> load(ncta);
    auto ffd = [&](long long cap) {
      std::fill(load.begin(), load.end(), 0);
      for (size_t i = 0; i < n; ++i) {
        int c = 0;
        while (c < ncta && load[c] + w[i].first > cap) ++c;
        if (c == ncta) return false;
        load[c] += w[i].first;
        fit[i] = c;
      }
      return true;
    };
    while (hi - lo > 1) {
      const long long mid = lo + (hi - lo) / 2;
      if (ffd(mid)) {
        hi = mid;
        fit_best = fit;
      } else {
        lo = mid;
      }
    }
    if (!fit_best.empty() && hi * 100 <= best * 97) bin = fit_best;
  }
  std::vector<std::vector<U>> lists(ncta);
  for (size_t i = 0; i < n; ++i) lists[bin[i]].push_back(w[i].second);
  units.clear();
  off.assign(ncta + 1, 0);
  for (int c = 0; c < ncta; ++c) {
    off[c] = (int)units.size();
    units.insert(units.end(), lists[c].begin(), lists[c].end());
  }
  off[ncta] = (int)units.size();
  if (cta_cost) {
    cta_cost->assign(ncta, 0);
    for (size_t i = 0; i < n; ++i) (*cta_cost)[bin[i]] += w[i].first;
  }
}

// The same deal by groups of units (grp[i]: group of unit i; equal ids come in
// runs, in order): the groups are dealt one after the other, each group's
// units by decreasing cost to the least-loaded CTA, and every CTA runs its
// units group by group, heaviest first within a group.  With a KV head per
// group, the units of one head are in flight on most CTAs at the same time,
// so the query tiles they walk (and the dQ rows they add into) are shared
// through L2 instead of coming from DRAM once per CTA.  (Keeping the plain
// deal and only running each CTA's units head by head does not do it: the
// CTAs drift apart across heads.  Measured on the MLA layer: backward 168 ms
// that way against 116 ms dealt by head.)
template <typename U>
void plan_units_grouped(std::vector<std::pair<long long, U>> w, const std::vector<int>& grp, int num_sms,
                        std::vector<U>& units, std::vector<int>& off, std::vector<long long>* cta_cost = nullptr) {
  const int ncta = (int)std::min<size_t>(w.size(), (size_t)std::max(1, num_sms));
  using Load = std::pair<long long, int>;  // (cost so far, CTA): ties go to the lower CTA
  std::priority_queue<Load, std::vector<Load>, std::greater<Load>> pq;
  for (int c = 0; c < ncta; ++c) pq.push({0, c});
  std::vector<std::vector<U>> lists(ncta);
  // The smallest units, whose costs add up to at least one largest unit per
  // CTA, are held back and dealt last, all groups together, heaviest first:
  // they even out what the grouped phase leaves (even where a group's costs
  // are far apart, e.g. one shard's units of a sequence's first and last
  // chunks), at the price of head order for a small share of the work.
  long long cut = -1;
  {
    std::vector<long long> c(w.size());
    long long mx = 0;
    for (size_t i = 0; i < w.size(); ++i) {
      c[i] = w[i].first;
      mx = std::max(mx, c[i]);
    }
    std::sort(c.begin(), c.end());
    long long acc = 0;
    for (size_t i = 0; i < c.size() && acc < mx * ncta; ++i) {
      acc += c[i];
      cut = c[i];
    }
  }
  auto deal = [&](std::vector<std::pair<long long, U>>& seg) {
    std::stable_sort(seg.begin(), seg.end(), [](const auto& x, const auto& y) { return x.first > y.first; });
    for (const auto& cu : seg) {
      const Load top = pq.top();
      pq.pop();
      lists[top.second].push_back(cu.second);
      pq.push({top.first + cu.first, top.second});
    }
  };
  std::vector<std::pair<long long, U>> seg, tail;
  for (size_t i0 = 0; i0 < w.size();) {
    size_t i1 = i0;
    while (i1 < w.size() && grp[i1] == grp[i0]) ++i1;
    seg.clear();
    for (size_t i = i0; i < i1; ++i) (w[i].first <= cut ? tail : seg).push_back(w[i]);
    deal(seg);
    i0 = i1;
  }
  deal(tail);
  if (cta_cost) {
    cta_cost->assign(ncta, 0);
    while (!pq.empty()) {
      (*cta_cost)[pq.top().second] = pq.top().first;
      pq.pop();
    }
  }
  units.clear();
  off.assign(ncta + 1, 0);
  for (int c = 0; c < ncta; ++c) {
    off[c] = (int)units.size();
    units.insert(units.end(), lists[c].begin(), lists[c].end());
  }
  off[ncta] = (int)units.size();
}

template <typename U>
int upload_plan(std::vector<std::pair<long long, U>> w, int num_sms, UnitPlan<U>& plan,
                const std::vector<int>* grp = nullptr) {
  std::vector<U> units;
  std::vector<int> off;
  if (grp) plan_units_grouped(std::move(w), *grp, num_sms, units, off);
  else plan_units(std::move(w), num_sms, units, off);
  int rc = upload(plan.units, units);
  if (!rc) rc = upload(plan.off, off);
  plan.ncta = (int)off.size() - 1;
  return rc;
}

// ---- argument checks ------------------------------------------------------
constexpr int kTile = 128;  // rows per attention tile
constexpr int kMaxCache = 1 << 30;  // decode cache positions (lengths plus a slice stay in int range)

int check_attn(const AttnShape& sh) {
  if (sh.B < 1 || sh.S < 1 || sh.Hq < 1 || sh.Hkv < 1 || sh.cp < 1)
    return fail(CPATTN_ERR_INVALID_ARG, "B, S, Hq, Hkv and cp must be >= 1");
  if (sh.Hq % sh.Hkv) return fail(CPATTN_ERR_INVALID_ARG, "Hq (%d) must be a multiple of Hkv (%d)", sh.Hq, sh.Hkv);
  if (sh.S % sh.cp) return fail(CPATTN_ERR_INVALID_ARG, "S (%d) must be a multiple of cp (%d)", sh.S, sh.cp);
  if (sh.lb < 0 || sh.lb > 2) return fail(CPATTN_ERR_INVALID_ARG, "load_balance must be 0, 1 or 2");
  if (sh.lb && sh.S % (2 * sh.cp))
    return fail(CPATTN_ERR_INVALID_ARG, "load balance needs S (%d) to be a multiple of 2*cp (%d)", sh.S, 2 * sh.cp);
  if (sh.lb == 2 && sh.cp > 1 && (sh.S / (2 * sh.cp)) % kTile)
    return fail(CPATTN_ERR_UNSUPPORTED, "zero-copy load balance needs the chunk length S/(2cp) = %d to be a multiple of %d",
                sh.S / (2 * sh.cp), kTile);
  const bool dims_ok = (sh.Dqk == 64 && sh.Dv == 64) || (sh.Dqk == 128 && sh.Dv == 128) ||
                       (sh.Dqk == 192 && sh.Dv == 128);
  if (!dims_ok)
    return fail(CPATTN_ERR_UNSUPPORTED, "head dims (Dqk=%d, Dv=%d) not in {(64,64),(128,128),(192,128)}", sh.Dqk,
                sh.Dv);
  if ((long long)sh.B * sh.S * sh.Hq > (1LL << 31) - 1)
    return fail(CPATTN_ERR_UNSUPPORTED, "B*S*Hq exceeds 2^31");
  return CPATTN_OK;
}

int check_ptrs(std::initializer_list<const void*> ps) {
  for (const void* p : ps) {
    if (!p) return fail(CPATTN_ERR_INVALID_ARG, "null tensor pointer");
    if (!aligned16(p)) return fail(CPATTN_ERR_INVALID_ARG, "tensor pointer %p is not 16-byte aligned", p);
  }
  return CPATTN_OK;
}

// ---- work lists ------------------------------------------------------------

int count_kv_tiles(const PosMap& pm, int bound) {
  int n = 0;
  for (int kt = next_kv_tile(pm, kTile, -1, bound); kt >= 0; kt = next_kv_tile(pm, kTile, kt, bound)) ++n;
  return n;
}
int tile_max_pos(const PosMap& pm, int t, int T) {
  int mn, mx;
  pm.range(t * T, t * T + T, mn, mx);
  return mx;
}
int tile_min_pos(const PosMap& pm, int t, int T) {
  int mn, mx;
  pm.range(t * T, t * T + T, mn, mx);
  return mn;
}

// The grouped deal (by KV head), only with many units per CTA (with few, the
// plain deal's MULTIFIT packing matters more).  The plain deal runs units of
// equal cost together, i.e. the same tile index of every head, so B*Hkv heads
// share the SMs.  Forward: always (measured: the DeepSeek-V3-shaped MLA layer,
// 128 KV heads, 47 -> 37 ms; the Llama3.1-70B-shaped layer, 8 KV heads,
// 205 -> 198 ms).  Backward: only where the plain deal leaves each head on
// fewer than about four CTAs (B*Hkv >= 64): the MLA backward gains a third
// from it, but the 70B-shaped backward loses 6% (152 CTAs then add into the
// same head's dQ rows at once, where the plain deal spreads them over 8).
bool use_grouped_deal(const AttnShape& sh, size_t n_units, int num_sms, bool backward) {
  if (n_units <= (size_t)std::max(1, num_sms) * 8) return false;
  return !backward || (long long)sh.B * sh.Hkv >= 64;
}

// forward units: pairs of 128-row query tiles sharing a KV head, with their
// cost (query tiles x (key steps + 4 steps of per-unit overhead))
std::vector<std::pair<long long, FwdUnit>> build_fwd_units(const AttnShape& sh, int shard,
                                                           std::vector<int>* grp = nullptr) {
  const PosMap pm = PosMap::make(sh.S, sh.cp, sh.lb);
  const int nqt = (sh.S + kTile - 1) / kTile;
  const int G = sh.Hq / sh.Hkv;
  const int per = sh.S / sh.cp;
  auto in_shard = [&](int qt) { return shard < 0 || (qt * kTile >= shard * per && qt * kTile < (shard + 1) * per); };
  std::vector<int> qmax(nqt);
  for (int qt = 0; qt < nqt; ++qt) qmax[qt] = tile_max_pos(pm, qt, kTile);
  std::vector<std::pair<long long, FwdUnit>> w;
  auto add = [&](int b, int hkv, int h0, int t0, int h1, int t1) {
    int bound = qmax[t0];
    if (h1 >= 0) bound = std::max(bound, qmax[t1]);
    const int nkv = count_kv_tiles(pm, bound);
    FwdUnit u{b, h0, h1, t0, t1, hkv, nkv, 0};
    const long long cost = (long long)(nkv + 4) * (h1 >= 0 ? 2 : 1);
    w.push_back({cost, u});
    if (grp) grp->push_back(b * sh.Hkv + hkv);
  };
  // tiles of one head paired with their neighbour in the same memory chunk
  auto pair_rows = [&](int b, int hkv, int h) {
    int qt = 0;
    while (qt < nqt) {
      if (!in_shard(qt)) { ++qt; continue; }
      const bool same_chunk = !pm.lb || (pm.c % kTile != 0) || ((qt * kTile) / pm.c == ((qt + 1) * kTile) / pm.c);
      if (qt + 1 < nqt && in_shard(qt + 1) && same_chunk) {
        add(b, hkv, h, qt, h, qt + 1);
        qt += 2;
      } else {
        add(b, hkv, h, qt, -1, 0);
        qt += 1;
      }
    }
  };
  for (int b = 0; b < sh.B; ++b)
    for (int hkv = 0; hkv < sh.Hkv; ++hkv) {
      const int h_first = hkv * G;
      int i = 0;
      for (; i + 1 < G; i += 2)  // two heads of the group on the same rows
        for (int qt = 0; qt < nqt; ++qt)
          if (in_shard(qt)) add(b, hkv, h_first + i, qt, h_first + i + 1, qt);
      if (i < G) pair_rows(b, hkv, h_first + i);
    }
  return w;
}

int fwd_units_cached(DevState& ds, const AttnShape& sh, int shard, UnitPlan<FwdUnit>** out) {
  std::vector<int> key{sh.B, sh.Hq, sh.Hkv, sh.S, sh.cp, sh.lb, shard};
  auto it = ds.fwd_units.find(key);
  if (it == ds.fwd_units.end()) {
    UnitPlan<FwdUnit> plan;
    std::vector<int> grp;
    auto w = build_fwd_units(sh, shard, &grp);
    const bool grouped = use_grouped_deal(sh, w.size(), ds.num_sms, false);
    int rc = upload_plan(std::move(w), ds.num_sms, plan, grouped ? &grp : nullptr);
    if (rc) return rc;
    it = ds.fwd_units.emplace(key, plan).first;
  }
  *out = &it->second;
  return CPATTN_OK;
}

// backward units.  kind 0: dk/dv, one 128-row key tile of a KV head, cost =
// query tiles (of BQ rows, all heads of the group) that see it; for one
// shard (shard >= 0) only the query tiles that hold a slot of the shard
// count, and key tiles none of them sees are left out, so the shard's launch
// is dealt by its own work.  kind 1: dq, one 128-row query tile of a query
// head, cost = key tiles it sees.  Both plus 3 steps of per-unit overhead.
int bwd_units_cached(DevState& ds, const AttnShape& sh, int kind, UnitPlan<BwdUnit>** out, int shard = -1) {
  std::vector<int> key{kind, sh.B, sh.Hq, sh.Hkv, sh.S, sh.cp, sh.lb, sh.Dqk, shard};
  auto it = ds.bwd_units.find(key);
  if (it == ds.bwd_units.end()) {
    const PosMap pm = PosMap::make(sh.S, sh.cp, sh.lb);
    const int nt = (sh.S + kTile - 1) / kTile;
    std::vector<std::pair<long long, BwdUnit>> w;
    std::vector<int> grp;  // kind 0: the KV head of each unit, for the grouped deal
    if (kind == 0) {
      const int BQ = bwd_dkdv_q_tile(sh.Dqk);
      const int lo = shard < 0 ? 0 : shard * (sh.S / sh.cp), hi = shard < 0 ? sh.S : (shard + 1) * (sh.S / sh.cp);
      std::vector<long long> cost(nt, -1);
      for (int kt = 0; kt < nt; ++kt) {
        const int bound = tile_min_pos(pm, kt, kTile);
        long long n = 0;
        for (int qt = next_q_tile(pm, BQ, -1, bound); qt >= 0; qt = next_q_tile(pm, BQ, qt, bound))
          if (qt * BQ < hi && qt * BQ + BQ > lo) ++n;
        if (n == 0 && shard >= 0) continue;
        cost[kt] = n + 3;
      }
      for (int b = 0; b < sh.B; ++b)
        for (int g = 0; g < sh.Hkv; ++g)
          for (int kt = 0; kt < nt; ++kt)
            if (cost[kt] >= 0) {
              w.push_back({cost[kt], BwdUnit{b, g, kt, 0}});
              grp.push_back(b * sh.Hkv + g);
            }
    } else {
      const int BK = bwd_dq_kv_tile(sh.Dqk);
      const int lo = shard < 0 ? 0 : shard * (sh.S / sh.cp), hi = shard < 0 ? sh.S : (shard + 1) * (sh.S / sh.cp);
      for (int qt = 0; qt < nt; ++qt) {
        if (qt * kTile >= hi || qt * kTile + kTile <= lo) continue;  // no slot of the shard
        const int bound = tile_max_pos(pm, qt, kTile);
        long long n = 0;
        for (int kt = next_kv_tile(pm, BK, -1, bound); kt >= 0; kt = next_kv_tile(pm, BK, kt, bound)) ++n;
        for (int b = 0; b < sh.B; ++b)
          for (int h = 0; h < sh.Hq; ++h) w.push_back({n + 3, BwdUnit{b, h, qt, 0}});
      }
    }
    const bool grouped = kind == 0 && use_grouped_deal(sh, w.size(), ds.num_sms, true);
    UnitPlan<BwdUnit> plan;
    int rc = upload_plan(std::move(w), ds.num_sms, plan, grouped ? &grp : nullptr);
    if (rc) return rc;
    it = ds.bwd_units.emplace(key, plan).first;
  }
  *out = &it->second;
  return CPATTN_OK;
}

int permute_impl(const void* src, void* dst, int B, int S, long long row_bytes, int cp, int inverse,
                 cudaStream_t st) {
  if (!src || !dst) return fail(CPATTN_ERR_INVALID_ARG, "null pointer");
  if (src == dst) return fail(CPATTN_ERR_INVALID_ARG, "src and dst must differ (the reorder is not in place)");
  if (B < 1 || S < 1 || cp < 1 || row_bytes < 1) return fail(CPATTN_ERR_INVALID_ARG, "B, S, cp, row_bytes must be >= 1");
  if (S % (2 * cp)) return fail(CPATTN_ERR_INVALID_ARG, "S (%d) must be a multiple of 2*cp (%d)", S, 2 * cp);
  const long long total = (long long)B * S * row_bytes;
  const char* s8 = static_cast<const char*>(src);
  const char* d8 = static_cast<const char*>(dst);
  if (s8 < d8 + total && d8 < s8 + total) return fail(CPATTN_ERR_INVALID_ARG, "src and dst overlap");
  std::lock_guard<std::mutex> lk(g_mu);
  DevState* ds;
  int rc = get_state(&ds);
  if (rc) return rc;
  cudaError_t e;
  {
    ProfScope ps(inverse ? "lb_unpermute" : "lb_permute", st);
    e = launch_lb_permute(src, dst, B, S, row_bytes, cp, inverse, ds->num_sms, st);
  }
  if (e != cudaSuccess) return cuda_fail(e, "lb_permute launch");
  return CPATTN_OK;
}

// test hook of the bounded waits: consumed by the next forward launch
struct FwdStall {
  int stage = -1;
  long long limit = 0;
};
FwdStall g_fwd_stall;

// k_rope non-null: MLA with one rope key per token shared by the heads (k holds
// the per-head 128-column nope keys)
int fwd_impl(const void* q, const void* k, const void* v, void* out, float* lse, const AttnShape& sh, int shard,
             cudaStream_t st, const void* k_rope = nullptr) {
  int rc = check_attn(sh);
  if (rc) return rc;
  if ((rc = check_ptrs({q, k, v, out, lse}))) return rc;
  if (shard >= sh.cp) return fail(CPATTN_ERR_INVALID_ARG, "shard %d out of range [0, %d)", shard, sh.cp);
  std::lock_guard<std::mutex> lk(g_mu);
  DevState* ds;
  if ((rc = get_state(&ds))) return rc;
  if ((rc = need_sm103(*ds))) return rc;
  UnitPlan<FwdUnit>* plan;
  if ((rc = fwd_units_cached(*ds, sh, shard, &plan))) return rc;
  if (plan->units.n == 0) return CPATTN_OK;
  FwdArgs a{};
  if ((rc = make_tmap(&a.tq, q, sh.B, sh.S, sh.Hq, sh.Dqk, 128))) return rc;
  if ((rc = make_tmap(&a.tk, k, sh.B, sh.S, sh.Hkv, k_rope ? 128 : sh.Dqk, 128))) return rc;
  if ((rc = make_tmap(&a.tv, v, sh.B, sh.S, sh.Hkv, sh.Dv, 128))) return rc;
  if (k_rope && (rc = make_tmap(&a.tkr, k_rope, sh.B, sh.S, 1, 64, 128))) return rc;
  a.rope_shared = k_rope ? 1 : 0;
  a.out = out;
  a.lse = lse;
  a.units = plan->units.ptr;
  a.cta_off = plan->off.ptr;
  a.n_units = (int)plan->units.n;
  a.sh = sh;
  a.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)sh.Dqk));
  a.err = ds->err;
  a.wait_limit = kWaitLimitCycles;
  a.fault_skip_stage = -1;
  if (g_fwd_stall.stage >= 0) {
    a.fault_skip_stage = g_fwd_stall.stage;
    a.wait_limit = g_fwd_stall.limit;
    g_fwd_stall = FwdStall{};
  }
  const int grid = plan->ncta;
  cudaError_t e;
  {
    ProfScope ps(shard < 0 ? "attn_fwd" : "attn_fwd_shard", st);
    e = launch_attn_fwd(a, grid, st);
  }
  if (e != cudaSuccess) return cuda_fail(e, "attn_fwd launch");
  return CPATTN_OK;
}

}  // namespace

extern "C" {

int cp_lb_permute(const void* src, void* dst, int B, int S, long long row_bytes, int cp, cudaStream_t stream) {
  return permute_impl(src, dst, B, S, row_bytes, cp, 0, stream);
}

int cp_lb_unpermute(const void* src, void* dst, int B, int S, long long row_bytes, int cp, cudaStream_t stream) {
  return permute_impl(src, dst, B, S, row_bytes, cp, 1, stream);
}

int cp_attn_fwd(const void* q, const void* k, const void* v, void* out, float* lse, int B, int Hq, int Hkv, int S,
                int Dqk, int Dv, int cp, int load_balance, cudaStream_t stream) {
  AttnShape sh{B, Hq, Hkv, S, Dqk, Dv, cp, load_balance};
  return fwd_impl(q, k, v, out, lse, sh, -1, stream);
}

int cp_attn_fwd_shard(const void* q, const void* k, const void* v, void* out, float* lse, int B, int Hq, int Hkv,
                      int S, int Dqk, int Dv, int cp, int load_balance, int shard, cudaStream_t stream) {
  if (shard < 0) return fail(CPATTN_ERR_INVALID_ARG, "shard must be >= 0");
  AttnShape sh{B, Hq, Hkv, S, Dqk, Dv, cp, load_balance};
  return fwd_impl(q, k, v, out, lse, sh, shard, stream);
}

namespace {
// shard < 0: the whole backward; else only query slots [shard*S/cp, (shard+1)*S/cp)
// take part and dk/dv (optional, bf16) and dk_part/dv_part (fp32) get their partial sums
// k_rope non-null: MLA with shared rope keys (k and dk hold the per-head nope
// columns, dk_rope the rope gradient summed over heads)
int bwd_impl(const void* q, const void* k, const void* v, const void* out, const float* lse, const void* dout,
             void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int S, int Dqk, int Dv, int cp,
             int load_balance, int shard, float* dk_part, float* dv_part, cudaStream_t stream,
             const void* k_rope = nullptr, void* dk_rope = nullptr) {
  AttnShape sh{B, Hq, Hkv, S, Dqk, Dv, cp, load_balance};
  int rc;
  DevState* ds;
  if ((rc = get_state(&ds))) return rc;
  if ((rc = need_sm103(*ds))) return rc;
  const int Spad = (S + kTile - 1) / kTile * kTile;
  const size_t nstat = (size_t)B * Hq * Spad;
  if ((rc = ensure(ds->bwd_stats, 2 * nstat, stream, false))) return rc;
  // MLA head dims take their own fused kernel (per-shard calls keep the two-kernel path)
  const bool mla_fused = Dqk == 192 && Dv == 128 && shard < 0;
  const bool fused = bwd_fused_supported(Dqk, Dv) || mla_fused;
  const size_t nacc = (size_t)B * S * Hq * Dqk;
  if (fused && (rc = ensure(ds->dq_acc, nacc, stream, false))) return rc;
  UnitPlan<BwdUnit>* u_kv;
  UnitPlan<BwdUnit>* u_q = nullptr;
  if ((rc = bwd_units_cached(*ds, sh, 0, &u_kv, shard))) return rc;
  if (!fused && (rc = bwd_units_cached(*ds, sh, 1, &u_q, shard))) return rc;
  BwdArgs a{};
  a.lse_l2 = ds->bwd_stats.ptr;
  a.delta = ds->bwd_stats.ptr + nstat;
  a.dq_acc = fused ? ds->dq_acc.ptr : nullptr;
  a.dq = dq;
  a.dk = dk;
  a.dv = dv;
  a.q_lo = shard < 0 ? 0 : shard * (S / cp);
  a.q_hi = shard < 0 ? S : (shard + 1) * (S / cp);
  a.dk_part = dk_part;
  a.dv_part = dv_part;
  a.Spad = Spad;
  a.sh = sh;
  a.scale = (float)(1.0 / std::sqrt((double)Dqk));
  a.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)Dqk));
  a.err = ds->err;
  cudaError_t e;
  {
    ProfScope ps("bwd_preprocess", stream);
    e = launch_bwd_preprocess(out, dout, lse, const_cast<float*>(a.lse_l2), const_cast<float*>(a.delta), a.dq_acc,
                              sh, Spad, stream);
  }
  if (e != cudaSuccess) return cuda_fail(e, "bwd preprocess launch");
  if (shard >= 0) {  // key tiles (and query rows) the shard does not touch stay zero
    const size_t nk = (size_t)B * S * Hkv;
    cudaError_t ez = cudaSuccess;
    if (dk_part) ez = cudaMemsetAsync(dk_part, 0, nk * Dqk * sizeof(float), stream);
    if (ez == cudaSuccess && dv_part) ez = cudaMemsetAsync(dv_part, 0, nk * Dv * sizeof(float), stream);
    if (ez == cudaSuccess && dk) ez = cudaMemsetAsync(dk, 0, nk * Dqk * 2, stream);
    if (ez == cudaSuccess && dv) ez = cudaMemsetAsync(dv, 0, nk * Dv * 2, stream);
    if (ez == cudaSuccess && !fused) ez = cudaMemsetAsync(dq, 0, nacc * 2, stream);
    if (ez != cudaSuccess) return cuda_fail(ez, "clearing the shard partials");
  }
  const size_t nrope = (size_t)B * S * 64;
  if (k_rope) {
    if ((rc = ensure(ds->rope_acc, nrope, stream, false))) return rc;
    e = cudaMemsetAsync(ds->rope_acc.ptr, 0, nrope * sizeof(float), stream);
    if (e != cudaSuccess) return cuda_fail(e, "clearing the rope-key gradient");
    a.rope_shared = 1;
    a.dk_rope_acc = ds->rope_acc.ptr;
  }
  const int kcols = k_rope ? 128 : Dqk;
  if (fused) {
    // one kernel: 128-row key tiles, 128-row query steps (MLA: 64-row half-steps);
    // dQ through the fp32 accumulator
    const int qrows = mla_fused ? 64 : 128;
    if ((rc = make_tmap(&a.tq, q, B, S, Hq, Dqk, qrows))) return rc;
    if ((rc = make_tmap(&a.tdo, dout, B, S, Hq, Dv, qrows))) return rc;
    if ((rc = make_tmap(&a.tk, k, B, S, Hkv, kcols, 128))) return rc;
    if ((rc = make_tmap(&a.tv, v, B, S, Hkv, Dv, 128))) return rc;
    if (k_rope && (rc = make_tmap(&a.tkr, k_rope, B, S, 1, 64, 128))) return rc;
    if ((rc = make_tmap_f32(&a.tdq, a.dq_acc, B, S, Hq, Dqk, qrows))) return rc;
    a.units = u_kv->units.ptr;
    a.cta_off = u_kv->off.ptr;
    a.n_units = (int)u_kv->units.n;
    if (u_kv->ncta > 0) {
      ProfScope ps(mla_fused ? "attn_bwd_mla" : "attn_bwd_fused", stream);
      e = mla_fused ? launch_attn_bwd_mla(a, u_kv->ncta, stream) : launch_attn_bwd_fused(a, u_kv->ncta, stream);
    }
    if (e != cudaSuccess) return cuda_fail(e, "fused bwd launch");
    {
      ProfScope ps("bwd_dq_round", stream);
      e = PosMap::make(S, cp, load_balance).lb == 2 ? launch_bwd_dq_round_nat(a.dq_acc, dq, sh, a.scale, stream)
                                                     : launch_bwd_dq_round(a.dq_acc, dq, (long long)nacc, a.scale, stream);
    }
    if (e != cudaSuccess) return cuda_fail(e, "dq rounding launch");
    if (k_rope) {
      ProfScope ps("bwd_dq_round", stream);
      e = launch_bwd_dq_round(ds->rope_acc.ptr, dk_rope, (long long)nrope, 1.0f, stream);
      if (e != cudaSuccess) return cuda_fail(e, "rope-key gradient rounding launch");
    }
    return CPATTN_OK;
  }
  // dk/dv: key tiles of 128 rows, query/dout boxes of BQ rows
  const int BQ = bwd_dkdv_q_tile(Dqk);
  if ((rc = make_tmap(&a.tq, q, B, S, Hq, Dqk, BQ))) return rc;
  if ((rc = make_tmap(&a.tdo, dout, B, S, Hq, Dv, BQ))) return rc;
  if ((rc = make_tmap(&a.tk, k, B, S, Hkv, kcols, 128))) return rc;
  if ((rc = make_tmap(&a.tv, v, B, S, Hkv, Dv, 128))) return rc;
  if (k_rope && (rc = make_tmap(&a.tkr, k_rope, B, S, 1, 64, 128))) return rc;
  a.units = u_kv->units.ptr;
  a.cta_off = u_kv->off.ptr;
  a.n_units = (int)u_kv->units.n;
  if (u_kv->ncta > 0) {
    ProfScope ps(shard < 0 ? "attn_bwd_dkdv" : "attn_bwd_dkdv_shard", stream);
    e = launch_attn_bwd_dkdv(a, u_kv->ncta, stream);
  }
  if (e != cudaSuccess) return cuda_fail(e, "bwd dk/dv launch");
  // dq: query tiles of 128 rows, key/value boxes of BK rows
  const int BK = bwd_dq_kv_tile(Dqk);
  if ((rc = make_tmap(&a.tq, q, B, S, Hq, Dqk, 128))) return rc;
  if ((rc = make_tmap(&a.tdo, dout, B, S, Hq, Dv, 128))) return rc;
  if ((rc = make_tmap(&a.tk, k, B, S, Hkv, kcols, BK))) return rc;
  if ((rc = make_tmap(&a.tv, v, B, S, Hkv, Dv, BK))) return rc;
  if (k_rope && (rc = make_tmap(&a.tkr, k_rope, B, S, 1, 64, BK))) return rc;
  a.units = u_q->units.ptr;
  a.cta_off = u_q->off.ptr;
  a.n_units = (int)u_q->units.n;
  if (u_q->ncta > 0) {
    ProfScope ps(shard < 0 ? "attn_bwd_dq" : "attn_bwd_dq_shard", stream);
    e = launch_attn_bwd_dq(a, u_q->ncta, stream);
  }
  if (e != cudaSuccess) return cuda_fail(e, "bwd dq launch");
  if (k_rope) {
    ProfScope ps("bwd_dq_round", stream);
    e = launch_bwd_dq_round(ds->rope_acc.ptr, dk_rope, (long long)nrope, 1.0f, stream);
    if (e != cudaSuccess) return cuda_fail(e, "rope-key gradient rounding launch");
  }
  return CPATTN_OK;
}
}  // namespace

int cp_attn_bwd(const void* q, const void* k, const void* v, const void* out, const float* lse, const void* dout,
                void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int S, int Dqk, int Dv, int cp,
                int load_balance, cudaStream_t stream) {
  AttnShape sh{B, Hq, Hkv, S, Dqk, Dv, cp, load_balance};
  int rc = check_attn(sh);
  if (rc) return rc;
  if ((rc = check_ptrs({q, k, v, out, lse, dout, dq, dk, dv}))) return rc;
  std::lock_guard<std::mutex> lk(g_mu);
  return bwd_impl(q, k, v, out, lse, dout, dq, dk, dv, B, Hq, Hkv, S, Dqk, Dv, cp, load_balance, -1, nullptr,
                  nullptr, stream);
}

int cp_attn_bwd_shard(const void* q, const void* k, const void* v, const void* out, const float* lse,
                      const void* dout, void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int S, int Dqk,
                      int Dv, int cp, int load_balance, int shard, float* dk_part, float* dv_part,
                      cudaStream_t stream) {
  AttnShape sh{B, Hq, Hkv, S, Dqk, Dv, cp, load_balance};
  int rc = check_attn(sh);
  if (rc) return rc;
  if (shard < 0 || shard >= cp) return fail(CPATTN_ERR_INVALID_ARG, "shard %d outside [0, %d)", shard, cp);
  if (sh.lb == 2) return fail(CPATTN_ERR_UNSUPPORTED, "the per-shard backward takes tensors in slot order (load_balance 0 or 1)");
  if ((rc = check_ptrs({q, k, v, out, lse, dout, dq, dk_part, dv_part}))) return rc;
  if ((dk && (rc = check_ptrs({dk}))) || (dv && (rc = check_ptrs({dv})))) return rc;
  std::lock_guard<std::mutex> lk(g_mu);
  return bwd_impl(q, k, v, out, lse, dout, dq, dk, dv, B, Hq, Hkv, S, Dqk, Dv, cp, load_balance, shard, dk_part,
                  dv_part, stream);
}

int cp_attn_fwd_mla(const void* q, const void* k_nope, const void* k_rope, const void* v, void* out, float* lse,
                    int B, int H, int S, int cp, int load_balance, cudaStream_t stream) {
  int rc = check_ptrs({k_rope});
  if (rc) return rc;
  AttnShape sh{B, H, H, S, 192, 128, cp, load_balance};
  return fwd_impl(q, k_nope, v, out, lse, sh, -1, stream, k_rope);
}

int cp_attn_bwd_mla(const void* q, const void* k_nope, const void* k_rope, const void* v, const void* out,
                    const float* lse, const void* dout, void* dq, void* dk_nope, void* dk_rope, void* dv, int B, int H,
                    int S, int cp, int load_balance, cudaStream_t stream) {
  AttnShape sh{B, H, H, S, 192, 128, cp, load_balance};
  int rc = check_attn(sh);
  if (rc) return rc;
  if ((rc = check_ptrs({q, k_nope, k_rope, v, out, lse, dout, dq, dk_nope, dk_rope, dv}))) return rc;
  std::lock_guard<std::mutex> lk(g_mu);
  return bwd_impl(q, k_nope, v, out, lse, dout, dq, dk_nope, dv, B, H, H, S, 192, 128, cp, load_balance, -1, nullptr,
                  nullptr, stream, k_rope, dk_rope);
}

int gqa_decode(const void* q, const void* kcache, const void* vcache, const int* lens, void* out, int B, int Hq,
               int Hkv, int Smax, int D, cudaStream_t stream) {
  if (B < 1 || Hq < 1 || Hkv < 1 || Smax < 1) return fail(CPATTN_ERR_INVALID_ARG, "B, Hq, Hkv, Smax must be >= 1");
  if (Smax > kMaxCache) return fail(CPATTN_ERR_INVALID_ARG, "Smax (%d) above the supported %d", Smax, kMaxCache);
  if ((long long)B * Hkv * decode_max_split(Smax) > 0x7fffffffLL)
    return fail(CPATTN_ERR_INVALID_ARG, "B*Hkv*ceil(Smax/%d) exceeds 2^31 decode items", kDecodeSplit);
  if (Hq % Hkv) return fail(CPATTN_ERR_INVALID_ARG, "Hq (%d) must be a multiple of Hkv (%d)", Hq, Hkv);
  if (Hq / Hkv > 16) return fail(CPATTN_ERR_UNSUPPORTED, "Hq/Hkv = %d > 16", Hq / Hkv);
  if (D != 64 && D != 128) return fail(CPATTN_ERR_UNSUPPORTED, "decode head dim %d not in {64, 128}", D);
  if (!lens) return fail(CPATTN_ERR_INVALID_ARG, "null lens");
  int rc = check_ptrs({q, kcache, vcache, out});
  if (rc) return rc;
  std::lock_guard<std::mutex> lk(g_mu);
  DevState* ds;
  if ((rc = get_state(&ds))) return rc;
  if ((rc = need_sm103(*ds))) return rc;
  if ((rc = ensure(ds->dec_o, decode_part_o_floats(B, Hq, Hkv, Smax, D), stream, false))) return rc;
  if ((rc = ensure(ds->dec_ml, decode_part_ml_floats(B, Hq, Hkv, Smax), stream, false))) return rc;
  DecodeArgs a{};
  a.q = q; a.kc = kcache; a.vc = vcache; a.lens = lens; a.out = out;
  a.B = B; a.Hq = Hq; a.Hkv = Hkv; a.Smax = Smax; a.D = D;
  a.part_o = ds->dec_o.ptr; a.part_ml = ds->dec_ml.ptr; a.err = ds->err;
  cudaError_t e;
  {
    ProfScope ps("gqa_decode", stream);
    e = launch_gqa_decode(a, stream);
  }
  if (e != cudaSuccess) return cuda_fail(e, "gqa_decode launch");
  return CPATTN_OK;
}

int gqa_decode_int8(const void* q, const void* kcache, const void* vcache, const float* kscale,
                    const float* vscale, const int* lens, void* out, int B, int Hq, int Hkv, int Smax, int D,
                    cudaStream_t stream) {
  if (B < 1 || Hq < 1 || Hkv < 1 || Smax < 1) return fail(CPATTN_ERR_INVALID_ARG, "B, Hq, Hkv, Smax must be >= 1");
  if (Smax > kMaxCache) return fail(CPATTN_ERR_INVALID_ARG, "Smax (%d) above the supported %d", Smax, kMaxCache);
  if ((long long)B * Hkv * decode_max_split(Smax) > 0x7fffffffLL)
    return fail(CPATTN_ERR_INVALID_ARG, "B*Hkv*ceil(Smax/%d) exceeds 2^31 decode items", kDecodeSplit);
  if (Hq % Hkv) return fail(CPATTN_ERR_INVALID_ARG, "Hq (%d) must be a multiple of Hkv (%d)", Hq, Hkv);
  if (Hq / Hkv > 16) return fail(CPATTN_ERR_UNSUPPORTED, "Hq/Hkv = %d > 16", Hq / Hkv);
  if (D != 128) return fail(CPATTN_ERR_UNSUPPORTED, "int8 decode head dim %d is not 128", D);
  if (B > decode_int8_max_batch()) return fail(CPATTN_ERR_UNSUPPORTED, "int8 decode batch %d > %d", B, decode_int8_max_batch());
  if (!lens || !kscale || !vscale) return fail(CPATTN_ERR_INVALID_ARG, "null lens or scales");
  int rc = check_ptrs({q, kcache, vcache, out});
  if (rc) return rc;
  std::lock_guard<std::mutex> lk(g_mu);
  DevState* ds;
  if ((rc = get_state(&ds))) return rc;
  if ((rc = need_sm103(*ds))) return rc;
  if ((rc = ensure(ds->dec_o, decode_part_o_floats(B, Hq, Hkv, Smax, D), stream, false))) return rc;
  if ((rc = ensure(ds->dec_ml, decode_part_ml_floats(B, Hq, Hkv, Smax), stream, false))) return rc;
  DecodeArgs a{};
  a.q = q; a.kc = kcache; a.vc = vcache; a.lens = lens; a.out = out;
  a.kscale = kscale; a.vscale = vscale;
  a.B = B; a.Hq = Hq; a.Hkv = Hkv; a.Smax = Smax; a.D = D;
  a.part_o = ds->dec_o.ptr; a.part_ml = ds->dec_ml.ptr; a.err = ds->err;
  cudaError_t e;
  {
    ProfScope ps("gqa_decode_int8", stream);
    e = launch_gqa_decode(a, stream);
  }
  if (e != cudaSuccess) return cuda_fail(e, "gqa_decode_int8 launch");
  return CPATTN_OK;
}

int mla_decode(const void* q, const void* ckv, const int* lens, void* out, int B, int H, int Smax, float scale,
               cudaStream_t stream) {
  if (B < 1 || H < 1 || Smax < 1) return fail(CPATTN_ERR_INVALID_ARG, "B, H, Smax must be >= 1");
  if (H > 128) return fail(CPATTN_ERR_UNSUPPORTED, "mla_decode: H = %d > 128 heads", H);
  if (B > mla_decode_max_batch()) return fail(CPATTN_ERR_UNSUPPORTED, "mla_decode: batch %d > %d", B, mla_decode_max_batch());
  if (Smax > kMaxCache) return fail(CPATTN_ERR_INVALID_ARG, "Smax (%d) above the supported %d", Smax, kMaxCache);
  if (!(scale > 0.f) || !std::isfinite(scale)) return fail(CPATTN_ERR_INVALID_ARG, "scale must be positive and finite");
  if (!lens) return fail(CPATTN_ERR_INVALID_ARG, "null lens");
  int rc = check_ptrs({q, ckv, out});
  if (rc) return rc;
  std::lock_guard<std::mutex> lk(g_mu);
  DevState* ds;
  if ((rc = get_state(&ds))) return rc;
  if ((rc = need_sm103(*ds))) return rc;
  const int nch = mla_decode_chunks(Smax), nchp = (nch + 1) & ~1;
  if ((rc = ensure(ds->mla_o, (size_t)B * H * nch * 512, stream, false))) return rc;
  if ((rc = ensure(ds->mla_ml, (size_t)B * H * nchp * 2, stream, false))) return rc;
  MlaDecodeArgs a{};
  a.q = q; a.ckv = ckv; a.lens = lens; a.out = out;
  a.part_o = ds->mla_o.ptr; a.part_ml = ds->mla_ml.ptr; a.err = ds->err;
  a.B = B; a.H = H; a.Smax = Smax; a.nch = nch; a.nchp = nchp;
  a.scale_log2 = (float)(1.4426950408889634 * (double)scale);
  cudaError_t e;
  {
    ProfScope ps("mla_decode", stream);
    e = launch_mla_decode(a, ds->num_sms, stream);
  }
  if (e != cudaSuccess) return cuda_fail(e, "mla_decode launch");
  return CPATTN_OK;
}

int gqa_decode_noalloc(const void* q, const void* kcache, const void* vcache, const int* lens, void* out, int B,
                       int Hq, int Hkv, int Smax, int D, cudaStream_t stream) {
  if (B < 1 || Hq < 1 || Hkv < 1 || Smax < 1) return fail(CPATTN_ERR_INVALID_ARG, "B, Hq, Hkv, Smax must be >= 1");
  if (Smax > kMaxCache) return fail(CPATTN_ERR_INVALID_ARG, "Smax (%d) above the supported %d", Smax, kMaxCache);
  if ((long long)B * Hkv * decode_max_split(Smax) > 0x7fffffffLL)
    return fail(CPATTN_ERR_INVALID_ARG, "B*Hkv*ceil(Smax/%d) exceeds 2^31 decode items", kDecodeSplit);
  if (Hq % Hkv) return fail(CPATTN_ERR_INVALID_ARG, "Hq (%d) must be a multiple of Hkv (%d)", Hq, Hkv);
  if (Hq / Hkv > 16) return fail(CPATTN_ERR_UNSUPPORTED, "Hq/Hkv = %d > 16", Hq / Hkv);
  if (D != 64 && D != 128) return fail(CPATTN_ERR_UNSUPPORTED, "decode head dim %d not in {64, 128}", D);
  if (!lens) return fail(CPATTN_ERR_INVALID_ARG, "null lens");
  int rc = check_ptrs({q, kcache, vcache, out});
  if (rc) return rc;
  const size_t need = noalloc_decode_bytes(B, Hq, Hkv, Smax, D);
  if (need > noalloc_decode_limit())
    return fail(CPATTN_ERR_INVALID_ARG,
                "gqa_decode_noalloc: this shape needs %zu bytes of scratch, the fixed array holds %zu "
                "(use gqa_decode, or fewer sequences / a shorter cache)",
                need, noalloc_decode_limit());
  int dev = 0, major = 0, minor = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
  if (major != 10 || minor != 3)
    return fail(CPATTN_ERR_UNSUPPORTED, "this library is built for sm_103a (GB300); device is sm_%d%d", major, minor);
  e = launch_gqa_decode_noalloc(q, kcache, vcache, lens, out, B, Hq, Hkv, Smax, D, stream);
  if (e != cudaSuccess) return cuda_fail(e, "gqa_decode_noalloc");
  return CPATTN_OK;
}

int cp_lb_positions(int S, int cp, int load_balance, int* pos_host) {
  if (!pos_host) return fail(CPATTN_ERR_INVALID_ARG, "null pos_host");
  if (S < 1 || cp < 1) return fail(CPATTN_ERR_INVALID_ARG, "S and cp must be >= 1");
  if (load_balance && S % (2 * cp)) return fail(CPATTN_ERR_INVALID_ARG, "S must be a multiple of 2*cp");
  const PosMap pm = PosMap::make(S, cp, load_balance);
  for (int j = 0; j < S; ++j) pos_host[j] = pm.pos(j);
  return CPATTN_OK;
}

int cp_attn_tile_counts(int S, int cp, int load_balance, long long* per_shard_host) {
  if (!per_shard_host) return fail(CPATTN_ERR_INVALID_ARG, "null per_shard_host");
  if (S < 1 || cp < 1 || S % cp) return fail(CPATTN_ERR_INVALID_ARG, "need S >= 1, cp >= 1, S %% cp == 0");
  if (load_balance && S % (2 * cp)) return fail(CPATTN_ERR_INVALID_ARG, "S must be a multiple of 2*cp");
  const PosMap pm = PosMap::make(S, cp, load_balance);
  const int nqt = (S + kTile - 1) / kTile;
  const int per = S / cp;
  for (int s = 0; s < cp; ++s) per_shard_host[s] = 0;
  for (int qt = 0; qt < nqt; ++qt) {
    const int s = std::min(cp - 1, (qt * kTile) / per);
    per_shard_host[s] += count_kv_tiles(pm, tile_max_pos(pm, qt, kTile));
  }
  return CPATTN_OK;
}

int cp_attn_fwd_schedule(int B, int Hq, int Hkv, int S, int cp, int load_balance, int num_ctas,
                         long long* cta_cost_host) {
  return cp_attn_fwd_shard_schedule(B, Hq, Hkv, S, cp, load_balance, -1, num_ctas, cta_cost_host);
}

int cp_attn_fwd_shard_schedule(int B, int Hq, int Hkv, int S, int cp, int load_balance, int shard, int num_ctas,
                               long long* cta_cost_host) {
  if (!cta_cost_host) return fail(CPATTN_ERR_INVALID_ARG, "null cta_cost_host");
  if (num_ctas < 1) return fail(CPATTN_ERR_INVALID_ARG, "num_ctas must be >= 1");
  AttnShape sh{B, Hq, Hkv, S, 128, 128, cp, load_balance};
  int rc = check_attn(sh);
  if (rc) return rc;
  if (shard < -1 || shard >= cp) return fail(CPATTN_ERR_INVALID_ARG, "shard %d outside [-1, %d)", shard, cp);
  std::vector<FwdUnit> units;
  std::vector<int> off;
  std::vector<long long> cost;
  std::vector<int> grp;
  auto w = build_fwd_units(sh, shard, &grp);
  if (use_grouped_deal(sh, w.size(), num_ctas, false)) plan_units_grouped(std::move(w), grp, num_ctas, units, off, &cost);
  else plan_units(std::move(w), num_ctas, units, off, &cost);
  for (int c = 0; c < num_ctas; ++c) cta_cost_host[c] = c < (int)cost.size() ? cost[c] : 0;
  return CPATTN_OK;
}

int cp_attn_test_stall_forward(int stage, long long wait_limit_cycles) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (stage < 0) {
    g_fwd_stall = FwdStall{};
    return CPATTN_OK;
  }
  if (wait_limit_cycles < 100000 || wait_limit_cycles > kWaitLimitCycles)
    return fail(CPATTN_ERR_INVALID_ARG, "wait_limit_cycles must be in [1e5, %lld]", kWaitLimitCycles);
  g_fwd_stall.stage = stage;
  g_fwd_stall.limit = wait_limit_cycles;
  return CPATTN_OK;
}

int cp_attn_check_device(cudaStream_t stream) {
  std::lock_guard<std::mutex> lk(g_mu);
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  // the library's error word exists once a call that keeps scratch ran on this
  // device; looking for it creates nothing (so a caller of the allocation-free
  // decode alone may call this too)
  int word = 0;
  auto it = g_dev.find(dev);
  if (it != g_dev.end() && it->second.err) {
    e = cudaMemcpy(&word, it->second.err, sizeof(int), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpy(error word)");
    if (word != DEV_OK) cudaMemset(it->second.err, 0, sizeof(int));
  }
  int word_na = 0;  // the allocation-free decode keeps its own word in its static array
  e = noalloc_take_error(&word_na);
  if (e != cudaSuccess) return cuda_fail(e, "reading the allocation-free decode's error word");
  if (word == DEV_OK) word = word_na;
  if (word == DEV_OK) return CPATTN_OK;
  if (word == DEV_TIMEOUT) return fail(CPATTN_ERR_DEVICE_TIMEOUT, "a kernel pipeline wait timed out");
  if (word == DEV_LENS_CLAMPED) return fail(CPATTN_ERR_DEVICE_BOUNDS, "decode lens outside [0, Smax] were clamped");
  if (word == DEV_SMEM_ALIGN) return fail(CPATTN_ERR_CUDA, "a kernel's shared memory was not 1024-byte aligned");
  return fail(CPATTN_ERR_CUDA, "unknown device error %d", word);
}

int cp_attn_profile_start(void) {
  std::lock_guard<std::mutex> lk(g_mu);
  for (auto& r : g_prof) {
    g_ev_pool.push_back(r.a);
    g_ev_pool.push_back(r.b);
  }
  g_prof.clear();
  g_prof_on = true;
  return CPATTN_OK;
}

int cp_attn_profile_stop(cpattn_kernel_stat* stats, int max_stats, int* n_stats) {
  std::lock_guard<std::mutex> lk(g_mu);
  g_prof_on = false;
  if (!n_stats) return fail(CPATTN_ERR_INVALID_ARG, "null n_stats");
  std::vector<cpattn_kernel_stat> agg;
  for (auto& r : g_prof) {
    cudaError_t e = cudaEventSynchronize(r.b);
    if (e != cudaSuccess) return cuda_fail(e, "cudaEventSynchronize");
    float ms = 0.f;
    e = cudaEventElapsedTime(&ms, r.a, r.b);
    if (e != cudaSuccess) return cuda_fail(e, "cudaEventElapsedTime");
    cpattn_kernel_stat* hit = nullptr;
    for (auto& x : agg)
      if (std::string(x.name) == r.name) hit = &x;
    if (!hit) {
      cpattn_kernel_stat z{};
      snprintf(z.name, sizeof(z.name), "%s", r.name);
      agg.push_back(z);
      hit = &agg.back();
    }
    hit->launches += 1;
    hit->total_ms += ms;
    g_ev_pool.push_back(r.a);
    g_ev_pool.push_back(r.b);
  }
  g_prof.clear();
  *n_stats = (int)agg.size();
  for (int i = 0; i < (int)agg.size() && i < max_stats && stats; ++i) stats[i] = agg[i];
  return CPATTN_OK;
}

const char* cp_attn_last_error(void) { return g_last_error.c_str(); }

int cp_attn_release(void) {
  std::lock_guard<std::mutex> lk(g_mu);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return fail(CPATTN_ERR_CUDA, "cudaGetDevice failed");
  auto it = g_dev.find(dev);
  if (it == g_dev.end()) return CPATTN_OK;
  cudaDeviceSynchronize();
  DevState& s = it->second;
  for (auto& kv : s.fwd_units) { cudaFree(kv.second.units.ptr); cudaFree(kv.second.off.ptr); }
  for (auto& kv : s.bwd_units) { cudaFree(kv.second.units.ptr); cudaFree(kv.second.off.ptr); }
  cudaFree(s.bwd_stats.ptr);
  cudaFree(s.dq_acc.ptr);
  cudaFree(s.rope_acc.ptr);
  cudaFree(s.dec_o.ptr);
  cudaFree(s.dec_ml.ptr);
  cudaFree(s.mla_o.ptr);
  cudaFree(s.mla_ml.ptr);
  cudaFree(s.err);
  g_dev.erase(it);
  return CPATTN_OK;
}

}  // extern "C"
