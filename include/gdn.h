/*
 * gdn.h - C ABI of libgdn, the GB300 (sm_103a) Gated DeltaNet slot-pool step.
 *
 * The library runs the per-layer linear-attention step of a hybrid-attention
 * serving engine over a pool of recurrent-state slots.  Each slot holds one
 * request's GDN state: an fp32 SSM state per V head and a short convolution
 * history ("TokenSpeed" talk, section "为什么 Agentic 推理需要新推理引擎":
 * linear-attention state = SSM state + conv state).  Slots are working slots
 * (updated in place every decode step) or checkpoint slots (snapshot targets)
 * ("TokenSpeed alcanza 580 tps con Qwen3.5-397B-A17B en GPU", section "Ciclo
 * de vida de slots"); requests address them through integer slot ids (the
 * same page, section "Scheduler dual": mamba_pool_indices).
 *
 * Conventions for every call:
 *  - All pointers are DEVICE pointers owned by the caller.  The library keeps
 *    no state besides launch counters, allocates nothing and is thread-safe.
 *  - `stream` is a cudaStream_t (NULL = the legacy default stream).  Calls are
 *    asynchronous on it and never synchronise the host.
 *  - The returned gdn_status covers host-side argument checks and the launch
 *    itself.  Data-dependent problems (bad slot ids) are reported by OR-ing
 *    GDN_DEV_ERR_* bits into *dev_err (device memory, may be NULL); read it
 *    after synchronising the stream.  Kernels never trap.
 *  - Pools are updated in place; inputs are never written; outputs must not
 *    alias inputs.
 *  - Slot id -1 is padding: the row is skipped and its outputs are written as
 *    zeros.  Any other id outside [0, num_slots) is skipped the same way and
 *    sets GDN_DEV_ERR_SLOT_OOB.
 *
 * Layouts (row-major, C order):
 *   channels   C = 2*hk*dk + hv*dv, ordered q | k | v, each head-major
 *   pool.ssm   float [num_slots][hv][dv][dk]   (S transposed: dk contiguous)
 *   pool.conv  conv_dtype [num_slots][conv_width-1][C], oldest input first
 *   params.conv_w  float [C][conv_width]  (index conv_width-1 = newest input)
 *   params.A_log, params.dt_bias  float [hv]
 *   V head h reads QK head h / (hv/hk).
 *
 * The per-token arithmetic is the Gated DeltaNet step (Yang, Kautz &
 * Hatamizadeh, "Gated Delta Networks", ICLR 2025), which the pages name but
 * do not write out:
 *   y = SiLU(conv1d(history, x));  q,k,v = split(y)
 *   q^ = q / sqrt(|q|^2 + 1e-6) / sqrt(dk);  k^ = k / sqrt(|k|^2 + 1e-6)
 *   g = -exp(A_log) * softplus(a + dt_bias);  alpha = exp(g);  beta = sigmoid(b)
 *   S <- alpha (I - beta k^ k^T) S + beta k^ v^T;  o = S^T q^  (updated S)
 */
#ifndef GDN_H
#define GDN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* element types */
#define GDN_F32 0
#define GDN_BF16 1

typedef enum {
  GDN_OK = 0,
  GDN_ERR_INVALID_ARG = 1, /* null pointer, negative size, bad alignment, ... */
  GDN_ERR_UNSUPPORTED = 2, /* shape / dtype combination not compiled in      */
  GDN_ERR_CUDA = 3,        /* the launch failed (cudaGetLastError)            */
  GDN_ERR_SCRATCH_LIMIT = 4 /* needs more than the built-in static scratch   */
} gdn_status;

/* bits OR-ed into *dev_err by the kernels */
#define GDN_DEV_ERR_SLOT_OOB 1u /* a slot id (or accept length) out of range   */
#define GDN_DEV_ERR_TIMEOUT 2u  /* a bounded inter-CTA wait gave up            */
#define GDN_DEV_ERR_SEQLENS 4u  /* prefill: cu_seqlens / start_pos inconsistent */

typedef struct {
  int32_t hk;         /* QK heads                                   */
  int32_t hv;         /* V heads, a multiple of hk                  */
  int32_t dk;         /* key/query head dim: 16, 64 or 128          */
  int32_t dv;         /* value head dim: 1..256                     */
  int32_t conv_width; /* conv1d width W: 2..8                       */
  int32_t act_dtype;  /* GDN_F32 or GDN_BF16: qkv, a, b and outputs */
  int32_t conv_dtype; /* GDN_F32 or GDN_BF16: the conv history      */
} gdn_dims;

typedef struct {
  float* ssm;        /* [num_slots][hv][dv][dk], 16-byte aligned */
  void* conv;        /* [num_slots][conv_width-1][C]             */
  int32_t num_slots;
} gdn_pool;

typedef struct {
  const float* conv_w;  /* [C][conv_width] */
  const float* A_log;   /* [hv]            */
  const float* dt_bias; /* [hv]            */
} gdn_params;

/*
 * Decode: one token per request, state updated in place in its working slot
 * (TokenSpeed Qwen3.5 page, "Scheduler dual": the state is updated in place at
 * every decode step).  For each request r with slot s = slot_ids[r]:
 * causal conv1d update of the history, SiLU, q/k L2 norm, gates, gated delta
 * rule on every V head, readout from the updated state.
 *   slot_ids [B] int32, distinct (precondition)
 *   qkv [B][C], a [B][hv], b [B][hv]  (act_dtype)
 *   out [B][hv][dv] (act_dtype; bf16 is rounded to nearest even)
 * B = 0 is a no-op.
 */
gdn_status gdn_decode_step(const gdn_dims* dims, gdn_pool pool,
                           const gdn_params* params, const int32_t* slot_ids,
                           int32_t B, const void* qkv, const void* a,
                           const void* b, void* out, uint32_t* dev_err,
                           void* stream);

/*
 * KDA decode (TokenSpeed talk, "为什么 Agentic 推理需要新推理引擎": Kimi K3's KDA
 * is the second linear-attention family whose SSM + conv state the engine
 * keeps; the pages do not write it).  The published Kimi Delta Attention step:
 * the gated delta rule with one decay per key channel,
 *   S <- (I - beta k^ k^T) diag(alpha) S + beta k^ v^T,  o = S^T q^,
 *   alpha_c = exp(-exp(A_log[h]) * softplus(a[h][c] + dt_bias[h][c])),
 * over the same slot pool, conv history, q/k norms and beta as
 * gdn_decode_step.  Arguments as for gdn_decode_step except:
 *   a [B][hv][dk] (act_dtype): per-channel gate logits
 *   params->dt_bias [hv][dk] float
 */
gdn_status gdn_kda_decode_step(const gdn_dims* dims, gdn_pool pool,
                               const gdn_params* params, const int32_t* slot_ids,
                               int32_t B, const void* qkv, const void* a,
                               const void* b, void* out, uint32_t* dev_err,
                               void* stream);

/*
 * KDA speculative verify: gdn_spec_verify with every draft step the KDA step
 * of gdn_kda_decode_step (a [B][T][hv][dk] per-channel gate logits,
 * params->dt_bias [hv][dk]).  Snapshots have the pool layout, so
 * gdn_spec_commit and gdn_spec_commit_index apply unchanged.
 */
gdn_status gdn_kda_spec_verify(const gdn_dims* dims, gdn_pool work, gdn_pool spec,
                               const gdn_params* params, const int32_t* slot_ids,
                               const int32_t* spec_ids, int32_t B, int32_t T,
                               const void* qkv, const void* a, const void* b,
                               void* out, uint32_t* dev_err, void* stream);

/*
 * KDA prefill: the contract of gdn_chunk_prefill (packed sequences from any
 * start position, block-aligned checkpoints of SSM state and conv history,
 * final state into the working slot) with every token the KDA step of
 * gdn_kda_decode_step; a [total_tokens][hv][dk], params->dt_bias [hv][dk].
 * fp32 accuracy: dk = 128 with dv <= 128 runs a 16-token chunked form (its
 * products on the tensor cores in split tf32), other shapes the token
 * recurrence.  A zero decay on a key channel (a = +inf) is exact on both.
 * Needs no workspace; ckpt_block a positive multiple of 64.
 */
gdn_status gdn_kda_prefill(const gdn_dims* dims, gdn_pool pool, gdn_pool ckpt,
                           const gdn_params* params, const int32_t* slot_ids,
                           const int32_t* cu_seqlens, const int64_t* start_pos, int32_t n_seq,
                           int64_t total_tokens, const int32_t* ckpt_ids, int32_t max_ckpt,
                           int32_t ckpt_block, const void* qkv, const void* a, const void* b,
                           void* out, uint32_t* dev_err, void* stream);

/*
 * Speculative verify (TokenSpeed Qwen3.5 page, "Scheduler dual": spec_cache
 * of per-step conv/SSM snapshots for rollback).  Request r runs its T draft
 * tokens starting from working slot slot_ids[r], which is NOT modified; after
 * draft t the full slot state (SSM + conv history) is written into spec slot
 * spec_ids[r][t] of pool `spec` (-1: not written).
 *   spec_ids [B][T] int32, distinct, disjoint from the working slots if the
 *   two pools are the same memory (precondition); 1 <= T <= 16
 *   qkv [B][T][C], a,b [B][T][hv], out [B][T][hv][dv]
 */
gdn_status gdn_spec_verify(const gdn_dims* dims, gdn_pool work, gdn_pool spec,
                           const gdn_params* params, const int32_t* slot_ids,
                           const int32_t* spec_ids, int32_t B, int32_t T,
                           const void* qkv, const void* a, const void* b,
                           void* out, uint32_t* dev_err, void* stream);

/*
 * Commit after verification (same section: rollback when verification
 * rejects drafts).  accept_len[r] = L in 0..T: L >= 1 copies spec slot
 * spec_ids[r][L-1] into working slot slot_ids[r]; L = 0 leaves the working
 * slot as is (it already holds the pre-draft state).  L outside 0..T sets
 * GDN_DEV_ERR_SLOT_OOB and skips the request.
 */
gdn_status gdn_spec_commit(const gdn_dims* dims, gdn_pool spec, gdn_pool work,
                           const int32_t* spec_ids, const int32_t* accept_len,
                           const int32_t* slot_ids, int32_t B, int32_t T,
                           uint32_t* dev_err, void* stream);

/*
 * Chunked prefill with block-aligned checkpoints (TokenSpeed Qwen3.5 page,
 * "Ciclo de vida de slots": a checkpoint becomes reusable once filled with
 * clean state and attached to a block-aligned prefix node).  Sequence n owns
 * tokens [cu_seqlens[n], cu_seqlens[n+1]) of the packed inputs; its first
 * token sits at absolute position start_pos[n] and its state (read, then
 * replaced by the final state) is slot slot_ids[n] of `pool`.  For every
 * absolute position P with P % ckpt_block == 0 and
 * start_pos[n] < P <= start_pos[n] + len, the state after token P-1 (SSM and
 * the last W-1 raw inputs) is written to checkpoint slot
 * ckpt_ids[n][P/ckpt_block - floor(start_pos[n]/ckpt_block) - 1] of `ckpt`
 * (-1 or an index >= max_ckpt: skipped).  The intra-chunk work uses chunks
 * of 64 tokens aligned to absolute positions.  A token whose decay is 0
 * (a = +inf) wipes the state before its update, as in gdn_decode_step; the
 * chunk form floors each token's log decay at -1000 to keep it exact.
 *   cu_seqlens [n_seq+1] int32 (device): absolute row offsets, non-decreasing,
 *     0 <= cu_seqlens[0], cu_seqlens[n_seq] <= total_tokens (usually 0 and
 *     total_tokens; rows outside them are not written and do not affect the
 *     results); a sequence whose rows fall outside [0, total_tokens) (or
 *     with start_pos < 0) is skipped and sets GDN_DEV_ERR_SEQLENS
 *   start_pos [n_seq] int64 (device)
 *   ckpt_ids [n_seq][max_ckpt] int32; ckpt_block a positive multiple of 64;
 *     max_ckpt above 262,140 returns GDN_ERR_UNSUPPORTED
 *   qkv [total_tokens][C], a,b [total_tokens][hv], out [total_tokens][hv][dv]
 *   workspace: >= gdn_chunk_prefill_workspace_size(...) bytes, 256-aligned
 */
size_t gdn_chunk_prefill_workspace_size(const gdn_dims* dims, int32_t n_seq,
                                        int64_t total_tokens);
gdn_status gdn_chunk_prefill(const gdn_dims* dims, gdn_pool pool, gdn_pool ckpt,
                             const gdn_params* params, const int32_t* slot_ids,
                             const int32_t* cu_seqlens, const int64_t* start_pos,
                             int32_t n_seq, int64_t total_tokens,
                             const int32_t* ckpt_ids, int32_t max_ckpt,
                             int32_t ckpt_block, const void* qkv, const void* a,
                             const void* b, void* out, void* workspace,
                             size_t workspace_bytes, uint32_t* dev_err,
                             void* stream);

/*
 * Chunked prefill with the readout epilogue fused: the call of
 * gdn_chunk_prefill, except that `y` ([total_tokens][hv][dv], activation
 * dtype, device) receives the gated RMS norm of the readout (see
 * gdn_gated_rmsnorm: y = o / sqrt(mean(o^2) + eps) * weight * silu(z), the
 * Gated DeltaNet block's output normalisation and gate; z [total_tokens][hv][dv]
 * in the activation dtype, weight [dv] fp32) instead of the readout itself.
 * State, checkpoints and conv histories are those of gdn_chunk_prefill.
 * The tf32 tensor-core prefill (dk = dv = 128, width 4, bf16 activations and
 * history) normalises each chunk's fp32 readout before it leaves the chip (z
 * and weight 16-byte aligned); every other case runs gdn_chunk_prefill into y
 * and then gdn_gated_rmsnorm on y in place.  Statuses as gdn_chunk_prefill,
 * plus GDN_ERR_INVALID_ARG for a null z or weight or eps < 0.
 */
gdn_status gdn_chunk_prefill_gated(const gdn_dims* dims, gdn_pool pool, gdn_pool ckpt,
                                   const gdn_params* params, const int32_t* slot_ids,
                                   const int32_t* cu_seqlens, const int64_t* start_pos,
                                   int32_t n_seq, int64_t total_tokens,
                                   const int32_t* ckpt_ids, int32_t max_ckpt,
                                   int32_t ckpt_block, const void* qkv, const void* a,
                                   const void* b, const void* z, const float* weight,
                                   float eps, void* y, void* workspace,
                                   size_t workspace_bytes, uint32_t* dev_err, void* stream);

/*
 * Chunked prefill that allocates nothing.  The pages have no counterpart to
 * this call; it is a convenience of this library.
 *
 * gdn_chunk_prefill needs a device workspace from its caller.  Some callers
 * cannot allocate device memory at the point where they run a prefill: code
 * hosted by a framework that owns all device memory and hands its plugins
 * only input and output pointers, or a runtime that reserves its whole memory
 * budget at start-up and allows no later cudaMalloc (which can synchronise
 * the device and would eat into that budget).  This variant takes the same
 * arguments as gdn_chunk_prefill minus the workspace, and works in a scratch
 * buffer built into the library: a static device array of
 * GDN_NOALLOC_SCRATCH_BYTES (64 MiB) that every GPU which loads the library
 * holds until the process exits.  That covers about 2,000 tokens per call of
 * a 16 QK / 32 V head, dk = dv = 128 layer (33,024 bytes per token); split a
 * longer prefill into several calls - the state carries over in the slot.
 *  - A call whose gdn_chunk_prefill_workspace_size(...) exceeds the scratch
 *    returns GDN_ERR_SCRATCH_LIMIT and launches nothing.
 *  - Every call looks up the scratch's device address in the current
 *    device's context (cudaGetSymbolAddress), so a device reset or another
 *    context needs nothing from the caller.  The first call on a device also
 *    loads the library's device code there; make that first call before any
 *    stream capture.
 *  - Every call on a device shares the one buffer and finds the previous
 *    call's contents in it.  Nothing in it needs to start at zero: each call
 *    writes what it later reads.  Calls that can overlap on the GPU (streams
 *    with no ordering between them) race on the buffer; order them.
 */
#define GDN_NOALLOC_SCRATCH_BYTES (64u << 20)
gdn_status gdn_chunk_prefill_noalloc(const gdn_dims* dims, gdn_pool pool,
                                     gdn_pool ckpt, const gdn_params* params,
                                     const int32_t* slot_ids,
                                     const int32_t* cu_seqlens,
                                     const int64_t* start_pos, int32_t n_seq,
                                     int64_t total_tokens,
                                     const int32_t* ckpt_ids, int32_t max_ckpt,
                                     int32_t ckpt_block, const void* qkv,
                                     const void* a, const void* b, void* out,
                                     uint32_t* dev_err, void* stream);

/*
 * Mixed batch: decode requests and prefill continuations in one packed batch
 * (TokenSpeed talk, "Kernel: 让 MLA 真正跑满 GPU": agent turns append a few
 * hundred tokens after a prefix hit, so batches are variable-length with no
 * padding; TokenSpeed Qwen3.5 page, "Scheduler dual": decode updates the
 * working slot in place).  Decode-first layout: sequences 0 .. n_decode-1 are
 * single-token decode requests whose tokens are rows 0 .. n_decode-1 of qkv /
 * a / b / out (cu_seqlens[i] = i for i <= n_decode; precondition); they take
 * exactly the gdn_decode_step update (no checkpoints; their start_pos and
 * ckpt_ids rows are not read).  Sequences n_decode .. n_seq-1 take exactly the
 * gdn_chunk_prefill update from any start position (the first chunk may
 * begin anywhere inside a 64-token chunk), with rows indexed by their absolute
 * cu_seqlens offsets.  All arguments as for gdn_chunk_prefill; the workspace
 * size gdn_chunk_prefill_workspace_size(dims, n_seq, total_tokens) suffices.
 * 0 <= n_decode <= min(n_seq, total_tokens), else GDN_ERR_INVALID_ARG.  Slot
 * ids must be distinct across the whole batch (precondition).  One call, on
 * one stream, with no host synchronisation.  Where both halves take their
 * fast paths (dk = dv = 128, conv width 4, bf16 activations and history,
 * 16-byte aligned qkv, out and conv weights, G * dv <= 256) and there are
 * both decode requests and continuations, the whole batch is ONE launch: a
 * persistent kernel whose work queue holds the continuations' chains, the
 * decode requests and the continuations' conv histories; it keeps that queue
 * in the first 8 * (2 + n_seq - n_decode) bytes of the workspace (8-byte
 * aligned; left zero after the call, and nothing in it needs to be zero
 * before), so workspace may be smaller than the prefill's size there but not
 * smaller than that.  Otherwise the decode rows go to the decode kernel and
 * the continuations to the chunked prefill (up to three launches).  Both give
 * the same bits as gdn_decode_step and gdn_chunk_prefill called one after
 * the other.  GDN_MIXED=split (read on every call) forces the separate
 * launches.
 */
gdn_status gdn_mixed_step(const gdn_dims* dims, gdn_pool pool, gdn_pool ckpt,
                          const gdn_params* params, const int32_t* slot_ids,
                          const int32_t* cu_seqlens, const int64_t* start_pos,
                          int32_t n_seq, int32_t n_decode, int64_t total_tokens,
                          const int32_t* ckpt_ids, int32_t max_ckpt, int32_t ckpt_block,
                          const void* qkv, const void* a, const void* b, void* out,
                          void* workspace, size_t workspace_bytes, uint32_t* dev_err,
                          void* stream);

/*
 * Copy-on-write from a clean slot (TokenSpeed Qwen3.5 page, "Riesgo de
 * correctitud: estado obsoleto": a reused working slot is made safe by a copy
 * from a checkpoint known to be clean, or by explicit zeroing).
 * dst slot dst_ids[i] of `dst` <- src slot src_ids[i] of `src`, SSM and conv
 * history, bit for bit.  The pools must have the same dims.  dst_ids must be
 * distinct and, when src and dst are the same pool, disjoint from src_ids
 * (precondition).
 */
gdn_status gdn_slot_copy(const gdn_dims* dims, gdn_pool src, gdn_pool dst,
                         const int32_t* src_ids, const int32_t* dst_ids,
                         int32_t n, uint32_t* dev_err, void* stream);

/* Explicit zeroing of slots ids[0..n) (same section): SSM and conv <- +0. */
gdn_status gdn_slot_zero(const gdn_dims* dims, gdn_pool pool,
                         const int32_t* ids, int32_t n, uint32_t* dev_err,
                         void* stream);

/*
 * Index-update commit (TokenSpeed talk, "Kernel: 让 MLA 真正跑满 GPU": the
 * accepted state is adopted by updating an index, not by moving data; Qwen3.5
 * page, "Scheduler dual": rollback keeps the pre-draft working slot).  For
 * callers whose spec snapshots live in the working pool (gdn_spec_verify with
 * spec == work).  Nothing but indices moves.  For request r, L = accept_len[r]:
 *   L = 0: slot_ids[r] is kept; freed_ids[r][t] = spec_ids[r][t].
 *   1 <= L <= T with spec_ids[r][L-1] >= 0: slot_ids[r] <- spec_ids[r][L-1];
 *     freed_ids[r][0] = the previous working slot, freed_ids[r][1..T) = the
 *     other snapshots in draft order (slots the caller returns to its
 *     allocator; -1 entries of spec_ids pass through).
 *   anything else: GDN_DEV_ERR_SLOT_OOB, slot_ids[r] kept, freed_ids[r][*] = -1.
 *   spec_ids [B][T], accept_len [B], slot_ids [B] (read and written),
 *   freed_ids [B][T] (written); all int32 device arrays.
 */
gdn_status gdn_spec_commit_index(const int32_t* spec_ids, const int32_t* accept_len,
                                 int32_t* slot_ids, int32_t* freed_ids, int32_t B,
                                 int32_t T, uint32_t* dev_err, void* stream);

/*
 * State pack / unpack for moving slot states between engines (TokenSpeed
 * Qwen3.5 page, "Disaggregacion Prefill-Decode": slot ids -> offsets ->
 * contiguous blocks for the transfer; this is the device half, no network).
 * Record i of `staging` (gdn_state_record_bytes(dims) bytes each, 16-byte
 * aligned, n records) is slot ids[i]: its SSM (fp32 [hv][dv][dk]) followed by
 * its conv history ([W-1][C] in the conv dtype), byte for byte as in the pool.
 *   pack:   record i <- slot ids[i]; id -1 gives a zero record; an id outside
 *           the pool gives a zero record and GDN_DEV_ERR_SLOT_OOB.
 *   unpack: slot ids[i] <- record i; -1 skips; an id outside the pool skips
 *           and sets GDN_DEV_ERR_SLOT_OOB.  ids must be distinct (precondition).
 *   staging_bytes >= n * record bytes, else GDN_ERR_INVALID_ARG.
 */
size_t gdn_state_record_bytes(const gdn_dims* dims);
gdn_status gdn_state_pack(const gdn_dims* dims, gdn_pool pool, const int32_t* ids, int32_t n,
                          void* staging, size_t staging_bytes, uint32_t* dev_err, void* stream);
gdn_status gdn_state_unpack(const gdn_dims* dims, const void* staging, size_t staging_bytes,
                            gdn_pool pool, const int32_t* ids, int32_t n, uint32_t* dev_err,
                            void* stream);

/*
 * Readout epilogue: gated RMS norm.  Not written on the pages; the published
 * Gated DeltaNet block normalises each head's readout and gates it with the
 * SiLU of a separate projection z.  For every (token, V head) row o of dv
 * values:  y = o / sqrt(mean(o^2) + eps) * weight * silu(z).
 *   o, z, y  [n_tokens][hv][dv] in the activation dtype, device; y may be o
 *            (in place); any other overlap is undefined;
 *   weight   [dv] fp32, device, shared by the heads;  eps >= 0.
 * Applies to the outputs of any call above (decode, verify, prefill, mixed).
 * Statuses as above; n_tokens = 0 launches nothing.
 */
gdn_status gdn_gated_rmsnorm(const gdn_dims* dims, const void* o, const void* z,
                             const float* weight, float eps, int64_t n_tokens, void* y,
                             void* stream);

/*
 * Self-test of the device-side failure path: one CTA waits on a barrier phase
 * that nothing completes; the bounded wait gives up after the library's wait
 * limit (1 s), GDN_DEV_ERR_TIMEOUT is OR-ed into *dev_err (device, required)
 * and the kernel returns, leaving the context usable.  Every kernel of this
 * library that waits on another agent (a copy engine, a tensor-core product,
 * a producer warp) waits the same way.  GDN_ERR_INVALID_ARG when dev_err is
 * null.
 */
gdn_status gdn_selftest_wait_timeout(uint32_t* dev_err, void* stream);

/* Human-readable name of a status code (static string). */
const char* gdn_status_string(int32_t status);

/* Launch counters: how many kernels of each kind this process launched. */
#define GDN_K_DECODE 0
#define GDN_K_SPEC_VERIFY 1
#define GDN_K_SLOT_COPY 2
#define GDN_K_SLOT_ZERO 3
#define GDN_K_SPEC_COMMIT 4
#define GDN_K_PREFILL 5
#define GDN_K_COMMIT_INDEX 6
#define GDN_K_STATE_PACK 7 /* pack and unpack */
#define GDN_K_GATED_RMSNORM 8
#define GDN_K_KDA_DECODE 9
#define GDN_K_KDA_VERIFY 10
#define GDN_K_KDA_PREFILL 11 /* the recurrence and its conv-history kernel */
#define GDN_K_MIXED 12       /* the single-launch mixed step */
#define GDN_K_COUNT 13
uint64_t gdn_launch_count(int32_t kernel);
void gdn_launch_count_reset(void);

/*
 * Bounds words of the checked build (libgdn_debug.so, compiled with
 * GDN_DEBUG_BOUNDS): every computed global, shared-memory and TMEM index of
 * the kernels is checked against the extent of its buffer (the tensor shapes
 * this header states, the CTA's shared-memory layout, the TMEM columns); an
 * index outside is counted, the first one's place recorded, and the access
 * redirected to element 0 or skipped, without a trap.  This call waits for
 * the device (cudaDeviceSynchronize), then copies the words out and clears
 * them:
 *   *count  number of failed checks since the last call (host, required);
 *   where   if count > 0, "<source file>:<line> <global|shared|TMEM>" of the
 *           first failure in the first unit that had one, NUL-terminated,
 *           truncated to where_len bytes (host; may be NULL);
 *   *index, *limit  that failure's index (for a span: its end) and the
 *           extent it was checked against (host; may be NULL).
 * GDN_ERR_UNSUPPORTED from the normal library (nothing is checked there),
 * GDN_ERR_INVALID_ARG for a null count, GDN_ERR_CUDA if a copy fails.
 */
gdn_status gdn_debug_bounds_take(uint32_t* count, char* where, size_t where_len, int64_t* index,
                                 int64_t* limit);

/*
 * Positive control of the checked build: one kernel makes three out-of-range
 * requests that the checks must catch (an index one past a global view, one
 * past a shared view, a span ending past its view), each view covering only
 * half of its buffer so that nothing outside real memory is ever touched.  A
 * following gdn_debug_bounds_take() reports count 3, the first "global".
 * GDN_ERR_UNSUPPORTED from the normal library (launches nothing).
 */
gdn_status gdn_selftest_bounds(void* stream);

#ifdef __cplusplus
}
#endif
#endif /* GDN_H */
