// Launchers shared between the C-ABI layer (api.cu) and the kernel files.
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace cpattn {

cudaError_t launch_lb_permute(const void* src, void* dst, int B, int S, long long row_bytes, int cp,
                              int inverse, int num_sms, cudaStream_t st);

// split-K decode: scratch = partial (o, m, l) per 128-position slice; a
// second kernel merges the slices of each (batch, kv head).
// bf16 tiled tensor map, 128-byte swizzle (returns 0 on success)
int decode_int8_max_batch();
// tensor map with 128-byte swizzle and zero fill; elem_bytes 2 (bf16), 1 (int8 as bytes) or 4 (fp32)
int encode_tmap(CUtensorMap* m, const void* ptr, int rank, const unsigned long long* dims,
                const unsigned long long* strides, const unsigned* box, int elem_bytes);
int encode_bf16_tmap(CUtensorMap* m, const void* ptr, int rank, const unsigned long long* dims,
                     const unsigned long long* strides, const unsigned* box);

struct DecodeArgs {
  CUtensorMap tk, tv, tq;  // used by the tensor-core path (D = 128)
  CUtensorMap tk2, tv2;    // the same caches in 32-row boxes (short slices)
  const void* q;
  const void* kc;
  const void* vc;
  const int* lens;
  void* out;
  int B, Hq, Hkv, Smax, D;
  const float* kscale;  // int8 cache only: [B, Hkv, Smax] per-position scales (null: bf16 cache)
  const float* vscale;
  float* part_o;    // [B*Hkv][max_split][G][D]
  float* part_ml;   // [B*Hkv][max_split][G][2]
  int* err;
};
constexpr int kDecodeSplit = 128;  // cache positions per CTA
int decode_max_split(int Smax);
size_t decode_part_o_floats(int B, int Hq, int Hkv, int Smax, int D);
size_t decode_part_ml_floats(int B, int Hq, int Hkv, int Smax);
cudaError_t launch_gqa_decode(const DecodeArgs& a, cudaStream_t st);
// allocation-free decode: scratch in a fixed static device array
size_t noalloc_decode_bytes(int B, int Hq, int Hkv, int Smax, int D);
size_t noalloc_decode_limit();
cudaError_t launch_gqa_decode_noalloc(const void* q, const void* kc, const void* vc, const int* lens, void* out,
                                      int B, int Hq, int Hkv, int Smax, int D, cudaStream_t st);
// read and clear the allocation-free decode's error word on the current device
// (symbol copies only; 0 if that decode never ran there)
cudaError_t noalloc_take_error(int* word);

// absorbed-MLA decode: latent rows of 576 columns (512 compressed KV, then 64
// rope) shared by every head; value = the first 512 columns
struct MlaDecodeArgs {
  CUtensorMap tq, tk;
  const void* q;     // [B, H, 576] bf16
  const void* ckv;   // [B, Smax, 576] bf16
  const int* lens;   // [B]
  void* out;         // [B, H, 512] bf16
  float* part_o;     // [B][H][nch][512] fp32 chunk partials
  float* part_ml;    // [B][H][nchp][2] (row max in the log2 domain, row sum); nchp = nch rounded up to even
  int* err;
  int B, H, Smax, nch, nchp;
  float scale_log2;
};
int mla_decode_chunks(int Smax);  // 256-position chunks of a cache of Smax
int mla_decode_max_batch();
cudaError_t launch_mla_decode(const MlaDecodeArgs& a, int num_sms, cudaStream_t st);

// ---- attention ------------------------------------------------------------
struct AttnShape {
  int B, Hq, Hkv, S, Dqk, Dv, cp, lb;
};

// one forward work unit: two query tiles (qt, head) that share a KV head
struct FwdUnit {
  int b;
  int h0, h1;   // query heads of the two tiles; h1 < 0: single tile
  int t0, t1;   // query tile indices (128-slot tiles)
  int hkv;
  int nkv;      // key tiles the unit walks (each step holds one)
  int pad;
};

struct FwdArgs {
  CUtensorMap tq, tk, tv;
  // MLA with one rope key per token shared by all heads (Dqk = 192): tk maps
  // the per-head 128-column nope keys, tkr the [B, S, 1, 64] rope keys, which
  // fill K's third 64-column box
  CUtensorMap tkr;
  int rope_shared;
  void* out;
  float* lse;
  const FwdUnit* units;
  const int* cta_off;  // CTA c runs units [cta_off[c], cta_off[c+1])
  int n_units;
  AttnShape sh;
  float scale_log2;
  int* err;
  long long wait_limit;  // SM clock cycles a pipeline wait may take before it gives up
  int fault_skip_stage;  // test hook: the producer skips this ring stage's loads (-1: none)
};
cudaError_t launch_attn_fwd(const FwdArgs& a, int grid, cudaStream_t st);
int attn_fwd_smem_bytes(int Dqk, int Dv);

struct BwdUnit {  // dk/dv unit: one key tile of one KV head; dq unit: one query tile of one head
  int b, h, t, pad;
};
struct BwdArgs {
  CUtensorMap tq, tk, tv, tdo;  // dq kernel uses 128-row boxes; dkdv uses BQ-row boxes for q/do
  CUtensorMap tkr;              // MLA shared rope keys [B, S, 1, 64] (rope_shared; tk: nope keys)
  int rope_shared;
  float* dk_rope_acc;           // rope_shared: [B, S, 64] fp32, dK's rope columns summed over heads
  CUtensorMap tdq;              // fused kernel: fp32 dQ accumulator, 32-column x 128-row boxes
  float* dq_acc;                // fused kernel: [B, S, Hq, Dqk] fp32, zeroed by the preprocess
  int q_lo, q_hi;               // fused kernel: query slots that take part ([0, S) except per shard)
  float* dk_part;               // fused kernel, per shard: fp32 partial dk/dv (null: none)
  float* dv_part;
  const float* lse_l2;          // [B, Hq, Spad] -lse * log2(e), -inf in padding
  const float* delta;           // [B, Hq, Spad] -rowsum(dout*out), 0 in padding
  void* dq;
  void* dk;
  void* dv;
  const BwdUnit* units;
  const int* cta_off;  // CTA c runs units [cta_off[c], cta_off[c+1])
  int n_units;
  int Spad;
  AttnShape sh;
  float scale_log2;
  float scale;
  int* err;
};
cudaError_t launch_bwd_preprocess(const void* out, const void* dout, const float* lse, float* lse_l2,
                                  float* delta, float* dq_acc, const AttnShape& sh, int Spad, cudaStream_t st);
// fused backward (one kernel for dK, dV and dQ, the latter through an fp32
// accumulator) for Dqk == Dv in {64, 128}
bool bwd_fused_supported(int Dqk, int Dv);
cudaError_t launch_attn_bwd_fused(const BwdArgs& a, int grid, cudaStream_t st);
cudaError_t launch_bwd_dq_round(const float* acc, void* dq, long long n, float scale, cudaStream_t st);
// natural-order tensors (zero-copy load balance): the accumulator is in slot order
cudaError_t launch_bwd_dq_round_nat(const float* acc, void* dq, const AttnShape& sh, float scale, cudaStream_t st);
// fused backward for MLA head dims (Dqk = 192, Dv = 128): 64-row query
// half-steps, dQ through the fp32 accumulator (q/do/tdq maps of 64-row boxes)
cudaError_t launch_attn_bwd_mla(const BwdArgs& a, int grid, cudaStream_t st);
cudaError_t launch_attn_bwd_dkdv(const BwdArgs& a, int grid, cudaStream_t st);
cudaError_t launch_attn_bwd_dq(const BwdArgs& a, int grid, cudaStream_t st);
int bwd_dkdv_q_tile(int Dqk);  // query rows per step of the dk/dv kernel
int bwd_dq_kv_tile(int Dqk);   // key rows per step of the dq kernel

}  // namespace cpattn
