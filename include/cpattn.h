/*
 * cpattn -- load-balanced context-parallel causal attention and GQA decode
 * on GB300 (sm_103a).  C ABI of libcpattn.so.
 *
 * The method (MaxText pull request 1445 "Add context parallelism",
 * Description): keys and values are all-gathered, queries are sharded on
 * the sequence, and tokens are reordered so that every shard does about
 * the same attention work.  The sequence is cut into 2*cp chunks of
 * c = S/(2cp) tokens; shard s holds chunk s followed by chunk 2cp-1-s (for
 * cp = 2 and eight tokens: 0,1,6,7 | 2,3,4,5).  In memory the reordered
 * ("load-balanced", LB) sequence is the concatenation of the shards, so
 * memory slot j holds original position
 *     pos(j) = chunk(k)*c + (j mod c),   k = j / c,
 *     chunk(k) = k/2 for even k, 2cp-1-k/2 for odd k.
 * The attention mask is reordered with the tokens: the query in slot i
 * sees the key in slot j iff pos(j) <= pos(i).  All cp shards run on one
 * GPU as independent work units over the single gathered K/V; no
 * collective is involved.
 *
 * Tensor layouts (row-major, contiguous, every pointer 16-byte aligned):
 *   q    [B, S, Hq,  Dqk]  bf16      k  [B, S, Hkv, Dqk]  bf16
 *   v    [B, S, Hkv, Dv ]  bf16      out[B, S, Hq,  Dv ]  bf16
 *   lse  [B, Hq, S]        fp32 (natural-log logsumexp of the scaled scores)
 *   dq/dk/dv: bf16 with the shapes of q/k/v.
 * When load_balance = 1 every sequence-indexed tensor (q, k, v, out, lse,
 * dout, dq, dk, dv) is in LB slot order; cp_lb_permute produces it.
 * Query head h reads KV head h / (Hq/Hkv) (grouped-query attention; MLA is
 * the case Dqk = 192, Dv = 128 with Hq = Hkv).  scale = 1/sqrt(Dqk).
 *
 * Ownership: the caller owns every tensor.  All tensor pointers are DEVICE
 * pointers except where a parameter says "host".  Work lists and scratch
 * (backward row statistics, decode split partials) are allocated by the
 * library on first use per device and shape, cached, and freed by
 * cp_attn_release().
 *
 * Execution: every call is asynchronous on `stream` and never
 * synchronises.  Calls on one stream are ordered; the library keeps
 * per-device scratch, so concurrent calls on different streams of the same
 * device must not overlap (serialise them or use one stream).
 *
 * Errors: every call returns a cpattn_status.  A negative value means
 * nothing was launched; cp_attn_last_error() gives a message (thread
 * local).  Faults found on the device (a pipeline wait that timed out,
 * decode lengths outside [0, Smax]) are latched in a device error word and
 * returned by cp_attn_check_device().
 */
#ifndef CPATTN_H_
#define CPATTN_H_

#include <stdint.h>
#include <cuda_runtime.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  CPATTN_OK = 0,
  CPATTN_ERR_INVALID_ARG = -1,    /* bad pointer, size or alignment */
  CPATTN_ERR_UNSUPPORTED = -2,    /* valid but not implemented (head dims, GPU arch) */
  CPATTN_ERR_CUDA = -3,           /* a CUDA runtime/driver call failed */
  CPATTN_ERR_NO_MEMORY = -4,      /* scratch allocation failed */
  CPATTN_ERR_DEVICE_TIMEOUT = -5, /* a kernel's bounded pipeline wait ran out */
  CPATTN_ERR_DEVICE_BOUNDS = -6   /* decode lens[b] outside [0, Smax] (clamped) */
} cpattn_status;

/*
 * Load-balance reorder and its inverse ("Add context parallelism",
 * Description: the token reorder done with jnp.take).
 *   cp_lb_permute:   dst[b, j, :] = src[b, pos(j), :]
 *   cp_lb_unpermute: dst[b, pos(j), :] = src[b, j, :]
 * src, dst: device, [B, S, row_bytes] bytes, src != dst (not in place).
 * Requires S % (2*cp) == 0, cp >= 1, row_bytes >= 1.  The copy is
 * bit-exact for any element type.
 */
int cp_lb_permute(const void* src, void* dst, int B, int S, long long row_bytes, int cp,
                  cudaStream_t stream);
int cp_lb_unpermute(const void* src, void* dst, int B, int S, long long row_bytes, int cp,
                    cudaStream_t stream);

/*
 * Forward attention of all cp shards ("Add context parallelism",
 * Description: each shard's queries against the gathered K/V under the
 * reordered causal mask; "Add support for EP to context parallelism":
 * MHA and MLA head layouts).
 *   out = softmax(scale * q k^T + mask) v,  lse = ln sum exp(scale q k^T).
 * q, k, v: device inputs; out, lse: device outputs (overwritten).
 * load_balance: 0 = natural token order, no reorder; 1 = q, k, v (and out,
 * lse) in the load-balanced slot order that cp_lb_permute produces; 2 =
 * zero-copy: q, k, v, out, lse in natural token order, work split and mask
 * as for 1 (each 128-row tile of slots is read from and written to the rows
 * of its original positions, so no permute is needed; the same for
 * cp_attn_bwd's dout, dq, dk, dv).
 * Requires B >= 1, S >= 1, Hkv >= 1, Hq % Hkv == 0, S % cp == 0, with
 * load_balance 1 or 2 S % (2*cp) == 0, and with 2 (cp > 1) a chunk length
 * S/(2*cp) that is a multiple of 128 (else CPATTN_ERR_UNSUPPORTED).
 * (Dqk, Dv) in {(64,64), (128,128), (192,128)}.  Runs on tcgen05 tensor
 * cores; needs an sm_103 GPU.
 */
int cp_attn_fwd(const void* q, const void* k, const void* v, void* out, float* lse, int B, int Hq,
                int Hkv, int S, int Dqk, int Dv, int cp, int load_balance, cudaStream_t stream);

/*
 * Forward work of ONE shard only: writes the out/lse rows of the query
 * tiles that start inside slots [shard*S/cp, (shard+1)*S/cp).  Used to time
 * and check per-shard work.  Arguments as cp_attn_fwd plus 0 <= shard < cp.
 */
int cp_attn_fwd_shard(const void* q, const void* k, const void* v, void* out, float* lse, int B,
                      int Hq, int Hkv, int S, int Dqk, int Dv, int cp, int load_balance,
                      int shard, cudaStream_t stream);

/*
 * Backward of cp_attn_fwd (gradient of sum(out * dout)).
 *   D = rowsum(dout * out); P = exp(scale q k^T - lse); dv = P^T dout;
 *   dP = dout v^T; dS = P * (dP - D); dq = scale dS k; dk = scale dS^T q.
 * dk/dv sum over the query heads of a group and over all shards (the
 * transpose of the K/V all-gather).  q, k, v, out, lse, dout: device
 * inputs (out and lse as written by cp_attn_fwd); dq, dk, dv: device
 * outputs (overwritten).  Constraints as cp_attn_fwd.  With Dqk == Dv
 * (64 or 128) dq is summed in an fp32 scratch buffer of B*S*Hq*Dqk floats
 * (library-owned, grown on demand) by reduce-adds whose order varies, so
 * dq may differ in its last bits between calls; dk, dv are repeatable.
 */
int cp_attn_bwd(const void* q, const void* k, const void* v, const void* out, const float* lse,
                const void* dout, void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int S,
                int Dqk, int Dv, int cp, int load_balance, cudaStream_t stream);

/*
 * Backward work of ONE shard (the emulated reduce-scatter made visible):
 * only the query slots [shard*S/cp, (shard+1)*S/cp) take part.  Arguments as
 * cp_attn_bwd plus 0 <= shard < cp and two fp32 outputs:
 *   dq       bf16, device: full gradients on the shard's rows, zero elsewhere;
 *   dk_part, dv_part  fp32 [B, S, Hkv, Dqk|Dv], device: this shard's
 *            contribution (summing them over all shards gives dk, dv; keys
 *            no query of the shard sees get zero);
 *   dk, dv   bf16, device, may be NULL: the same partial sums rounded.
 * Head dims as cp_attn_bwd (the MLA dims run the two-kernel backward
 * restricted to the shard); load_balance 0 or 1 (slot-order tensors),
 * otherwise CPATTN_ERR_UNSUPPORTED.  Rows of a query tile that straddles a
 * shard boundary outside the shard are masked out, so the partials are
 * exact per shard for any S.
 */
int cp_attn_bwd_shard(const void* q, const void* k, const void* v, const void* out, const float* lse,
                      const void* dout, void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int S,
                      int Dqk, int Dv, int cp, int load_balance, int shard, float* dk_part,
                      float* dv_part, cudaStream_t stream);

/*
 * MLA with the rope key shared by all heads ("Add support for EP to context
 * parallelism in self-attention", Main code changes: MLA attention under
 * context parallelism; the shared rope key is the DeepSeek-V3 form of it):
 * each head's key is its own 128-column "nope" part followed by one 64-column
 * rope key per token that every head uses, so K is never materialised per
 * head.  The attention is exactly cp_attn_fwd / cp_attn_bwd with
 * Hq = Hkv = H, Dqk = 192, Dv = 128 and k[b, s, h] = concat(k_nope[b, s, h],
 * k_rope[b, s]); scale = 1/sqrt(192).
 *   q        bf16 [B, S, H, 192], device (nope columns, then rope columns)
 *   k_nope   bf16 [B, S, H, 128], device
 *   k_rope   bf16 [B, S, 64], device (one rope key per token)
 *   v        bf16 [B, S, H, 128], device
 *   out, lse as cp_attn_fwd (out [B, S, H, 128], lse fp32 [B, H, S]).
 * Order and load_balance as cp_attn_fwd; all token-indexed tensors in the
 * same order.
 */
int cp_attn_fwd_mla(const void* q, const void* k_nope, const void* k_rope, const void* v, void* out,
                    float* lse, int B, int H, int S, int cp, int load_balance, cudaStream_t stream);

/*
 * Backward of cp_attn_fwd_mla: dq [B, S, H, 192], dk_nope [B, S, H, 128],
 * dv [B, S, H, 128] as cp_attn_bwd, and dk_rope bf16 [B, S, 64] = the rope
 * columns of every head's dk summed over the heads (the gradient of the
 * shared rope key).  All outputs are device buffers, overwritten.  The rope
 * sum goes through an fp32 scratch buffer of B*S*64 floats (library-owned,
 * grown on demand) by atomic adds whose order varies, so dk_rope may differ
 * in its last bits between calls.
 */
int cp_attn_bwd_mla(const void* q, const void* k_nope, const void* k_rope, const void* v, const void* out,
                    const float* lse, const void* dout, void* dq, void* dk_nope, void* dk_rope, void* dv,
                    int B, int H, int S, int cp, int load_balance, cudaStream_t stream);

/*
 * Grouped-query decode attention ("Add Pallas GPU decode attention in
 * Maxtext inference", Description: decode attention through a GQA kernel):
 * one query token per sequence against a KV cache.
 *   out[b, h] = softmax_{t < lens[b]}(scale q[b,h] . kcache[b,g,t]) vcache[b,g,t],
 *   g = h / (Hq/Hkv), scale = 1/sqrt(D).
 * q [B, Hq, D] bf16, kcache/vcache [B, Hkv, Smax, D] bf16, lens [B] int32,
 * out [B, Hq, D] bf16; all device.  lens[b] == 0 gives out = 0; lens[b]
 * outside [0, Smax] is clamped and latched as CPATTN_ERR_DEVICE_BOUNDS.
 * Cache rows at or past lens[b] may be read but never reach the output.
 * Requires D in {64, 128}, Hq % Hkv == 0, Hq/Hkv <= 16, Smax <= 2^30.
 */
int gqa_decode(const void* q, const void* kcache, const void* vcache, const int* lens, void* out,
               int B, int Hq, int Hkv, int Smax, int D, cudaStream_t stream);

/*
 * Absorbed-MLA decode (MLA attention under context parallelism, "Add
 * support for EP to context parallelism in self-attention", Main code
 * changes, at decode time, "Add Pallas GPU decode attention in Maxtext
 * inference", Description): one query token per sequence; every head uses
 * the same cached latent row per token, 576 columns (the 512-column
 * compressed KV, then the 64-column rope key), as its key and the first
 * 512 columns of it as its value:
 *   out[b, h] = sum_{t < lens[b]} softmax_t(scale q[b,h] . ckv[b,t]) ckv[b,t,:512].
 * q [B, H, 576] bf16 (each head's query taken into the latent space, then
 * its rope query), ckv [B, Smax, 576] bf16, lens [B] int32, out [B, H, 512]
 * bf16 (the latent output, before the value up-projection); all device.
 * scale is the softmax scale of the attention the absorption comes from
 * (1/sqrt(192) for 128 nope + 64 rope columns).  lens[b] == 0 gives zeros;
 * lens outside [0, Smax] is clamped and latched as CPATTN_ERR_DEVICE_BOUNDS.
 * Cache rows at or past lens[b] are read but never reach the output.
 * Requires 1 <= H <= 128, B <= 1024, Smax <= 2^30.  Scratch: fp32 chunk
 * partials of B*ceil(Smax/256)*H*514 floats (library-owned, grown on demand).
 */
int mla_decode(const void* q, const void* ckv, const int* lens, void* out, int B, int H, int Smax, float scale,
               cudaStream_t stream);

/*
 * gqa_decode against an int8-quantised KV cache (the inference setup of
 * "rename context to context_autoregressive", Tests, runs with
 * quantize_kvcache=True): kcache/vcache int8 [B, Hkv, Smax, D], device, with
 * one fp32 scale per (batch, KV head, position) in kscale/vscale [B, Hkv,
 * Smax], device; the cached vector at position t is int8 values * scale.
 * The kernel dequantises each vector to bf16 (one rounding) and then runs
 * the tensor-core decode, reading half the bytes of the bf16 cache.  Other
 * arguments, layouts, results and error behaviour as gqa_decode.  Requires
 * D == 128, B <= 1024, Hq % Hkv == 0, Hq/Hkv <= 16.
 */
int gqa_decode_int8(const void* q, const void* kcache, const void* vcache, const float* kscale,
                    const float* vscale, const int* lens, void* out, int B, int Hq, int Hkv, int Smax,
                    int D, cudaStream_t stream);

/*
 * gqa_decode without any allocation by the library (the pages have no
 * counterpart; this exists for callers that must not let a library
 * allocate device memory: code whose memory is owned by a caching
 * allocator or a pool sized up front, serving loops that must avoid the
 * driver's allocation path and its implicit synchronisation, processes
 * that keep nearly all of HBM for their KV cache).
 * Same arguments, layouts and results as gqa_decode.  The split partials
 * live in one fixed 8 MiB device array inside the library (every GPU that
 * loads the library holds it until the process exits); the caller still
 * passes all inputs and outputs.  A shape whose scratch does not fit is
 * rejected with CPATTN_ERR_INVALID_ARG before any launch (about
 * B*Hkv*ceil(Smax/128)*G'*(D+2)*4 bytes, G' = Hq/Hkv rounded up to a power
 * of two; the decode workload B=24, Hkv=8, Smax=2048, G=4, D=128 needs
 * 6.1 MiB).
 * The first call on a device looks up the array's device address with that
 * device current; make that first call before any stream capture.  Every
 * call shares the one array (each call writes every entry it later reads,
 * so nothing an earlier call left behind is used), and calls whose
 * executions overlap on the GPU (different streams, or several host
 * threads) race on it: serialise them.  Device-side faults (lens outside
 * [0, Smax], clamped as in gqa_decode; a pipeline wait that timed out) are
 * latched in an error word inside the same array; cp_attn_check_device
 * reads and clears it with symbol copies, so checking allocates nothing
 * either.
 */
int gqa_decode_noalloc(const void* q, const void* kcache, const void* vcache, const int* lens,
                       void* out, int B, int Hq, int Hkv, int Smax, int D, cudaStream_t stream);

/* ---- helpers ---------------------------------------------------------- */

/* pos(j) for j in [0, S) into pos_host (host array of S ints). */
int cp_lb_positions(int S, int cp, int load_balance, int* pos_host);

/*
 * Work of each shard in (query tile, key tile) pairs of 128 x 128 slots
 * that the forward kernel visits per (batch, query head): per_shard_host
 * is a host array of cp long longs.  With load balance and c a multiple of
 * 128 every shard gets (2cp-1)m^2 + m(m+1) pairs, m = c/128.
 */
int cp_attn_tile_counts(int S, int cp, int load_balance, long long* per_shard_host);

/*
 * Host helper: the plan the forward uses on a GPU with num_ctas SMs.  The
 * forward's work units (pairs of 128-row query tiles sharing a KV head) are
 * dealt to min(units, num_ctas) CTAs so that the most-loaded CTA carries as
 * little as possible (with many units per CTA, one KV head after the other,
 * so that a head's units run on most SMs at the same time and share its K/V
 * tiles through L2); cta_cost_host[c] (host, num_ctas entries) receives the
 * modelled load of CTA c, a unit costing (its key steps + 4) per query tile it
 * holds; CTAs without units get 0.  Shapes as cp_attn_fwd (head dims do not
 * enter the plan).  No device work; returns CPATTN_OK or an argument error.
 */
int cp_attn_fwd_schedule(int B, int Hq, int Hkv, int S, int cp, int load_balance, int num_ctas,
                         long long* cta_cost_host);

/*
 * The same for the plan of one shard's forward (cp_attn_fwd_shard with that
 * shard); shard = -1 is the whole forward, as cp_attn_fwd_schedule.  Returns
 * CPATTN_OK or an argument error (shard outside [-1, cp)).
 */
int cp_attn_fwd_shard_schedule(int B, int Hq, int Hkv, int S, int cp, int load_balance, int shard, int num_ctas,
                               long long* cta_cost_host);

/*
 * Kernel timing for profiling and benchmarks.  Between profile_start and
 * profile_stop every kernel the library launches is bracketed by two CUDA
 * events recorded on its own stream.  profile_stop waits for those events
 * and fills `stats` (host array of max_stats entries, may be NULL) with one
 * entry per kernel name: launch count and summed device milliseconds;
 * *n_stats receives the number of distinct kernels.  Adds about two event
 * records per launch; off by default.
 */
typedef struct {
  char name[32];
  int launches;
  double total_ms;
} cpattn_kernel_stat;
int cp_attn_profile_start(void);
int cp_attn_profile_stop(cpattn_kernel_stat* stats, int max_stats, int* n_stats);

/*
 * Test hook for the bounded pipeline waits (no counterpart on the pages; it
 * exists so that the timeout path can be exercised without hanging a GPU).
 * The NEXT forward launch (cp_attn_fwd, cp_attn_fwd_shard or
 * cp_attn_fwd_mla on any thread) leaves out the loads of ring stage `stage`
 * in every CTA whose producer reaches that stage, and every pipeline wait
 * of that launch gives up after wait_limit_cycles SM clock cycles instead
 * of about two seconds.  The wait on the missing stage runs out, latches
 * CPATTN_ERR_DEVICE_TIMEOUT in the device error word (read it with
 * cp_attn_check_device), and every role of the CTA leaves its loop; the
 * launch ends with out/lse undefined and the device stays usable.
 * stage < 0 clears a pending hook.  Requires 1e5 <= wait_limit_cycles <= 4e9
 * when stage >= 0.
 */
int cp_attn_test_stall_forward(int stage, long long wait_limit_cycles);

/*
 * Synchronise `stream`, then read and clear the device error words of the
 * current device: the library's own (it exists once a call that keeps
 * scratch has run on the device; this call never creates it) and the
 * allocation-free decode's.  Returns CPATTN_OK, CPATTN_ERR_DEVICE_TIMEOUT or
 * CPATTN_ERR_DEVICE_BOUNDS; allocates no device memory.
 */
int cp_attn_check_device(cudaStream_t stream);

/* Thread-local message of the last failed call ("" if none). */
const char* cp_attn_last_error(void);

/* Free cached work lists and scratch of the current device. */
int cp_attn_release(void);

#ifdef __cplusplus
}
#endif
#endif /* CPATTN_H_ */
