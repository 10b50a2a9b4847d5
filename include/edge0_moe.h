/*
 * edge0_moe.h — C ABI of the latent-MoE layer library (libedge0_moe.so), B300 / sm_103a.
 *
 * The layer (one token; the pages' description):
 *   z = D x                       down-projection 2560 -> l, one D per layer
 *   l_e = R_e . z + b_e            router logits over the routed experts
 *   top-k experts by (logit desc, index asc), weights = softmax renormalised over the k
 *   o_e = W_d,e (silu(W_g,e z) * (W_up,e z))   each expert l -> 640 -> l, NVFP4 weights
 *   c = o_shared + sum_k w_k o_(e_k)           the shared expert runs alongside, weight 1
 *   y = U c                       up-projection l -> 2560, one U per layer
 * Sources: "Edge0-145B hardware requirements", section "Edge0-145B latent MoE
 * architecture: how 145B fits one GPU" (widths 2560 and 1792, 512 routed + 1
 * shared expert, 10 picked per token, D and U shared by the experts);
 * "Edge0-145B · Q3_K" model card, section "Architecture" (diagram caption:
 * D, router, experts l -> 640 -> l, shared expert, U; one D/U per layer;
 * config block: SwiGLU width 640); "Edge0 Squeezes a 145B Coding Agent...",
 * table "Released model variants" (latent 1792 for 145B, 1280 for 120B);
 * "Edge0-145B en local", introduction (experts in NVFP4, NVIDIA's 4-bit float).
 * The softmax/top-k rule, tie-break, NVFP4 record layout and this interface
 * are this library's readings; the pages print no formula or layout.
 *
 * Grouped latent projections (n_groups = G > 1; "Edge0-145B hardware
 * requirements", same section: eight groups of D and U per layer, each shared
 * by 64 experts, every expert labelled with its group; model card, section
 * "Architecture": D maps the token to the latent per routing group):
 *   z_g = D_g x for every group g;  l_e = R_e . z_(g(e)) + b_e
 *   expert e runs on z_(g(e)), the shared expert on z of shared_group
 *   c_g = [g = shared_group] o_shared + sum over kept k with g(e_k) = g of w_k o_(e_k)
 *   y = sum_g U_g c_g
 * With G = 1 this is the layer above.
 *
 * Conventions for every call:
 *   - Pointers named "device" point to CUDA device memory of the current device;
 *     "host" pointers to host memory.  The caller owns every buffer it passes.
 *   - Device pointers must be 16-byte aligned; expert records 256-byte aligned.
 *   - bf16 tensors are row-major arrays of IEEE bfloat16 (uint16 bit patterns).
 *   - Calls taking a stream are asynchronous with respect to the host, enqueue
 *     work on that stream (NULL = the legacy default stream) and do not
 *     synchronise, except where stated.
 *   - Errors are returned as edge0_status; nothing is printed and nothing exits.
 *     Asynchronous device-side failures (a bounded wait that ran out) are
 *     recorded in the handle's error word and reported by edge0_moe_get_error.
 */
#ifndef EDGE0_MOE_H
#define EDGE0_MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t; declared here so the header needs no CUDA headers. */
typedef struct CUstream_st *edge0_stream_t;

typedef enum {
  EDGE0_OK = 0,
  EDGE0_ERR_INVALID_ARG = 1,  /* bad pointer, size, shape or alignment */
  EDGE0_ERR_UNSUPPORTED = 2,  /* valid request the library does not support */
  EDGE0_ERR_CUDA = 3,         /* a CUDA runtime call failed */
  EDGE0_ERR_OOM = 4,          /* workspace allocation failed */
  EDGE0_ERR_TIMEOUT = 5       /* a device-side bounded wait ran out */
} edge0_status;

/*
 * NVFP4 expert record (one per expert, this library's layout).
 * Format (NVFP4 = E2M1 elements, one E4M3 scale per 16 consecutive weights
 * along the input dimension K, one fp32 scale g per matrix):
 *     w[r][k] = e2m1(code[r][k]) * e4m3(scale[r][k/16]) * g
 * For latent L (a multiple of 256) and SwiGLU width F (a multiple of 128) a
 * record holds, without gaps:
 *   GU block, F rows of 9L/8 bytes; row f =
 *       gate codes row f (L/2) | up codes row f (L/2) |
 *       gate scales row f (L/16) | up scales row f (L/16)
 *   D block, L/2 row pairs of 9F/8 bytes; pair p =
 *       down codes rows 2p, 2p+1 (F/2 each) | down scales rows 2p, 2p+1 (F/16 each)
 *   fp32 g: gate, up, down (little-endian)
 * W_gate, W_up are [F x L] (K = L); W_down is [L x F] (K = F).  Two codes per
 * byte, the even element in the low nibble.  E4M3 is OCP E4M3FN (bias 7,
 * subnormals m * 2^-9, no infinities; the NaN bytes 0x7F/0xFF must not occur).
 * Interleaving makes any run of gate/up rows, or of down row pairs, one
 * contiguous byte range, and every run starts on a 16-byte boundary.
 * For L=1792, F=640 the codes and scales take 1,935,360 bytes, the size that
 * 48 layers x 512 experts of the 47.6 GB NVFP4 experts.bin imply ("Edge0-145B
 * Review", table in section "Warum 29 GB nicht wirklich in 29 GB passen").
 */

/* Bytes of one record: codes + scales + 12 bytes of fp32 scales.  0 on bad shapes. */
size_t edge0_expert_record_bytes(int latent, int ffn);

/* Default distance between records in an array: record bytes rounded up to 256. */
size_t edge0_expert_record_stride(int latent, int ffn);

/*
 * Pack one expert from its per-matrix arrays into a record (host memory).
 * The per-matrix ("logical") arrays are row-major per matrix, concatenated:
 *   codes   host, 3*F*L/2 bytes: gate [F][L/2], up [F][L/2], down [L][F/2]
 *   scales  host, 3*F*L/16 bytes: gate [F][L/16], up [F][L/16], down [L][F/16]
 *   globals host, 3 floats: gate, up, down
 *   record_out host, edge0_expert_record_bytes(latent, ffn) bytes, caller-owned.
 * Returns INVALID_ARG on NULL pointers or unsupported shapes.
 */
edge0_status edge0_pack_expert_host(const uint8_t *codes, const uint8_t *scales,
                                    const float *globals, int latent, int ffn,
                                    void *record_out);

/*
 * Pack n_experts experts on the device (same per-expert arrays, back to back).
 *   codes    device, n_experts * 3*F*L/2 bytes
 *   scales   device, n_experts * 3*F*L/16 bytes
 *   globals  device, n_experts * 3 floats
 *   records  device, n_experts * stride bytes, 256-byte aligned; stride >=
 *            edge0_expert_record_bytes and a multiple of 16.
 * Bytes between a record's end and the next stride boundary are left untouched.
 */
edge0_status edge0_pack_experts(const uint8_t *codes, const uint8_t *scales,
                                const float *globals, int n_experts, int latent,
                                int ffn, void *records, size_t stride,
                                edge0_stream_t stream);

/*
 * Quantise an fp32 matrix to NVFP4 on the device (the format fixes the
 * decoder, not the quantiser; this is the plain reading):
 *   scale[r][b] = E4M3 round-to-nearest-even of amax(block) / (6 g), max 448;
 *   code[r][k]  = nearest E2M1 value to w / (e4m3(scale) g), ties to the even
 *                 code, saturating at +-6; an all-zero block gets scale 0.
 *   w       device fp32 [rows][K], K a multiple of 16
 *   codes   device uint8 [rows][K/2]; scales device uint8 [rows][K/16]
 */
edge0_status edge0_quantize_nvfp4(const float *w, int rows, int K, float g,
                                  uint8_t *codes, uint8_t *scales,
                                  edge0_stream_t stream);

/* One layer's shapes and borrowed device weights.  G = max(1, n_groups). */
typedef struct {
  int hidden;     /* 2560 */
  int latent;     /* l: 1792 (145B) or 1280 (120B); multiple of 256 */
  int n_experts;  /* 512 routed experts */
  int top_k;      /* 10 */
  int ffn;        /* SwiGLU width 640; multiple of 128 */
  int max_tokens; /* largest T forward will accept (workspace sizing) */
  const void *D;            /* device bf16 [G*latent][hidden]: rows g*latent.. are D_g */
  const void *U;            /* device bf16 [hidden][G*latent]: columns g*latent.. are U_g */
  const void *router;       /* device bf16 [n_experts][latent] */
  const float *router_bias; /* device fp32 [n_experts], or NULL for zeros */
  const void *experts;      /* device, n_experts records, 256-byte aligned */
  size_t expert_stride;     /* bytes between records; multiple of 256 */
  const void *shared_expert;/* device, one record, 256-byte aligned */
  int n_groups;             /* latent groups: 0 or 1 = one D/U pair; at most 16 */
  const int *expert_group;  /* G > 1: device int32 [n_experts], group of each routed
                               expert in [0, G); read once by edge0_moe_create */
  int shared_group;         /* G > 1: group of the shared expert, in [0, G) */
} edge0_moe_desc;

/*
 * Create a layer handle.  Validates shapes and alignment, records the
 * borrowed pointers (which must stay valid for the handle's lifetime) and
 * allocates the workspace for max_tokens (the handle owns only that).
 * Supported shapes: hidden % 64 == 0, latent % 256 == 0, ffn % 128 == 0,
 * ffn <= 1024, 1 <= top_k <= 16, top_k <= n_experts <= 1024, n_experts % 32 == 0, and
 * a decode shared-memory plan that fits the device (else UNSUPPORTED).  A grouped
 * layer (G > 1) also needs G * latent <= 16384, latent <= 2048 and valid labels
 * (else INVALID_ARG); it allocates workspace for max(max_tokens, 16) tokens.
 * Runs the router fold and the |z| bound on the device (legacy stream) and
 * synchronises before returning.
 * Returns INVALID_ARG, UNSUPPORTED, CUDA or OOM on failure (*handle_out = NULL).
 * Source: the layer's parts and widths, "Edge0-145B hardware requirements",
 * section "Edge0-145B latent MoE architecture: how 145B fits one GPU"; the D/U
 * groups and expert labels, the same section.
 */
edge0_status edge0_moe_create(const edge0_moe_desc *desc, void **handle_out);

/*
 * y = Layer(x) for T tokens.  x device bf16 [T][hidden]; y device bf16
 * [T][hidden] (round to nearest even); x and y must not overlap.
 * T = 0 is a no-op; T > max_tokens returns INVALID_ARG.  T <= 16 runs the
 * decode path (one persistent kernel); larger T the prefill path.  A grouped
 * layer (G > 1) runs the prefill path's kernels at every T.
 * Calls on one handle must be ordered (one stream, or synchronised): they
 * share the handle's workspace.
 * Source: the layer's steps (D, router, 10 of 512 experts l -> 640 -> l with a
 * shared expert, U), "Edge0-145B · Q3_K" model card, section "Architecture".
 */
edge0_status edge0_moe_forward(void *handle, const void *x, void *y, int T,
                               edge0_stream_t stream);

/*
 * Copy the routing of the last forward on this handle into caller buffers
 * (any may be NULL), stream-ordered after it:
 *   idx    device int32 [T][top_k], experts in rank order
 *   w      device fp32  [T][top_k], renormalised weights
 *   counts device int32 [n_experts], slots per expert
 *   offsets device int32 [n_experts + 1], exclusive prefix sum of counts
 *   perm   device int32 [T*top_k], slot (t*top_k + j) at each grouped position;
 *          groups in expert order, slots ascending within a group
 *   pos    device int32 [T*top_k], grouped position of each slot
 */
edge0_status edge0_moe_debug_routing(void *handle, int *idx, float *w, int *counts,
                                     int *offsets, int *perm, int *pos,
                                     edge0_stream_t stream);

/*
 * Copy an intermediate of the last forward (for stage-by-stage parity):
 *   what = 0: latent z [T][G*latent]; 1: router logits fp32 [T][n_experts];
 *   2: combined latent c [T][G*latent].  After a decode forward (T <= 16) z and
 *   c are fp32.  After a prefill forward (T > 16) they are in the form the
 *   experts and U consume: z as f16 z_t * 2^-e_t, with e_t the binary exponent
 *   of the bound max_r sum_h |D_rh| * max_h |x_t,h| (so every value is below 1
 *   in magnitude), and c as bf16.  After a prefill forward also what = 3: the
 *   SwiGLU activations H bf16 [T*top_k + T][ffn] and 4: the expert outputs O
 *   bf16 [T*top_k + T][latent], rows in grouped position order (the shared
 *   expert's T rows last).  A grouped layer's forwards are prefill forwards at
 *   every T.  dst device, `bytes` >= size.
 * Returns UNSUPPORTED if no forward has run yet, INVALID_ARG for other `what`.
 */
edge0_status edge0_moe_debug_tensor(void *handle, int what, void *dst, size_t bytes,
                                    edge0_stream_t stream);

/*
 * C = A B^T on the tensor cores (tcgen05, bf16 in, fp32 accumulate), the dense
 * GEMM the prefill path uses for D and U:
 *   A device bf16 [M][K] row-major, B device bf16 [N][K] row-major,
 *   C device fp32 [M][N] row-major (overwritten); K a multiple of 64.
 *   err   device int or NULL: a device wait that ran out ORs EDGE0_ERR_TIMEOUT's
 *         bit (1) into it (bounded waits; the kernel always finishes).
 */
edge0_status edge0_gemm_bf16_tn(const void *A, const void *B, float *C, int M, int N, int K,
                                int *err, edge0_stream_t stream);

/*
 * Post-norm residual between stacked layers (bf16 in, bf16 out):
 *   out[t] = bf16( v / sqrt(mean(v^2) + eps) ),  v = x[t] + y[t]  (fp32 inside)
 * x, y, out device bf16 [T][hidden]; out may alias x or y.
 */
edge0_status edge0_residual_rmsnorm(const void *x, const void *y, void *out, int T,
                                    int hidden, float eps, edge0_stream_t stream);

/*
 * Run n_layers layers in sequence with the post-norm residual between them:
 *   x_0 = x;  x_{i+1} = RMSNorm(x_i + Layer_i(x_i));  y = x_n
 * handles: host array of n_layers handles of identical shapes; T <= 16
 * (decode) runs all layers in one persistent kernel.  x, y device bf16
 * [T][hidden], may be the same buffer.  Larger T, or any grouped layer, chains
 * forward and edge0_residual_rmsnorm per layer.
 * The decode kernel reads a small device table of the layers, held by
 * handles[0]: a call with a list of layers different from the previous call's
 * uploads it (stream-ordered).  A call captured into a CUDA graph must use the
 * list of the preceding uncaptured call on handles[0]; otherwise it returns
 * EDGE0_ERR_UNSUPPORTED (the graph would reference host memory).
 * Source: 48 layers per model, model card "Edge0-145B · Q3_K", section
 * "Architecture" (config block); the residual norm between layers is this
 * library's reading (the pages give none).
 */
edge0_status edge0_moe_stack_forward(void *const *handles, int n_layers, const void *x,
                                     void *y, int T, float eps, edge0_stream_t stream);

/*
 * edge0_moe_stack_forward that also records every layer's input, output and
 * routing (for layer-by-layer checks): trace_x, trace_y device bf16
 * [n_layers][T][hidden]; trace_idx device int32 [n_layers][T][top_k], the
 * experts each layer kept for each token in rank order (any may be NULL).
 * Decode sizes of one-group layers only (T <= 16, n_layers <= 64, n_groups <= 1);
 * other calls return UNSUPPORTED when a trace is requested.
 */
edge0_status edge0_moe_stack_forward_trace(void *const *handles, int n_layers, const void *x,
                                           void *y, int T, float eps, void *trace_x,
                                           void *trace_y, int *trace_idx, edge0_stream_t stream);

/*
 * Decode forward (T <= 16) that allocates no device memory: the paper has no
 * counterpart; this entry exists for callers that cannot call cudaMalloc (a
 * host program that owns every device allocation and hands out a fixed budget,
 * a plug-in that may not grow the process's memory, a real-time loop where an
 * allocation or the synchronisation it can cause is not allowed).
 *   desc      the layer, as for edge0_moe_create (max_tokens is ignored)
 *   x, y      device bf16 [T][hidden], must not overlap
 *   status_out  device int or NULL: receives, stream-ordered after the forward,
 *             EDGE0_OK or the device error bits (a wait that ran out)
 * Scratch lives in one static device array of this library (about 7.8 MB, held
 * by every GPU that loads the library until the process exits).  Limits:
 * T <= 16, hidden <= 3072, latent <= 2048, n_experts <= 512, ffn <= 1024, one
 * latent group (n_groups 0 or 1), and the decode kernel's shared-memory plan
 * must fit the device (the check edge0_moe_create makes); other sizes return
 * EDGE0_ERR_UNSUPPORTED without launching anything.
 * The first call on a device looks up the array's device address and sets the
 * decode kernel's launch attributes (once per device, with that device
 * current): make that first call before any stream capture.  All calls share
 * the array and each clears the words that must start at zero; calls that
 * overlap on the GPU race, so the caller must serialise them.  Each call also
 * recomputes R D and the |z| bound max_r sum_h |D_rh| into the array (two
 * small kernels before the forward; the forward then scales z per token by a
 * power of two exactly as the handle path does).
 */
edge0_status edge0_moe_forward_noalloc(const edge0_moe_desc *desc, const void *x, void *y, int T,
                                       int *status_out, edge0_stream_t stream);

/*
 * Stage timing of the prefill path, for profiling.  While enabled, each
 * prefill forward on the handle records a CUDA event on its stream before its
 * first kernel and after each of its EDGE0_PREFILL_STAGES kernels:
 *   0 x -> [z | logits] GEMM, 1 top-k + chunk histogram, 2 chunk scan,
 *   3 expert offsets, 4 scatter, 5 z-row gather, 6 gate/up + SwiGLU grouped
 *   GEMM, 7 down grouped GEMM, 8 combine, 9 U GEMM.
 * edge0_moe_stage_times waits for the last forward's final event and writes
 * the n = min(max, EDGE0_PREFILL_STAGES) stage durations in milliseconds to
 * host ms[0..n); *n_out (if not NULL) = n.  UNSUPPORTED if the last forward
 * was not a timed prefill forward.  Enabling adds event records between the
 * kernels and nothing else; it is off by default.
 */
#define EDGE0_PREFILL_STAGES 10
edge0_status edge0_moe_profile_stages(void *handle, int enable);
edge0_status edge0_moe_stage_times(void *handle, float *ms, int max, int *n_out);

/*
 * Phase timing of the decode kernel, for profiling.  While enabled (the first
 * enable allocates a small stamp buffer on the handle), each decode forward or
 * stack call on the handle zeroes that buffer on its stream before the launch
 * and the kernel records %globaltimer stamps at its phase boundaries.
 * edge0_moe_decode_phase_times synchronises the device and writes, for each layer
 * of the last profiled launch, EDGE0_DECODE_PHASES microsecond values to host us[]:
 *   0 P0 (z and logits) on CTA 0's clock to the last CTA's end, 1 spread of the
 *   CTAs' P0 ends, 2 grid barrier 1, 3 routing (top-k, weights, permutation) on
 *   CTA 0, 4 rest of P1 (gate/up) to the last CTA's end, 5 spread of P1 ends,
 *   6 barrier 2, 7 P2 (down + combine), 8 spread, 9 barrier 3, 10 P3 (U), 11
 *   spread, 12 barrier 4 (stacks; 0 otherwise), 13 the layer's total; and on
 *   CTA 0's clock: 14 routing's loads of the logits and z, 15 the top-k and
 *   weights, 16 issue of the first expert copies after routing, 17 P2's first
 *   staging of h, 18 P2's down MMAs of all rounds.
 * n = min(max, layers * EDGE0_DECODE_PHASES); *n_out = n.  UNSUPPORTED if no
 * profiled decode launch ran.  Profiling adds one memset per launch and a few
 * stores per CTA and phase.
 */
#define EDGE0_DECODE_PHASES 19
edge0_status edge0_moe_profile_decode(void *handle, int enable);
edge0_status edge0_moe_decode_phase_times(void *handle, float *us, int max, int *n_out);

/*
 * Expert residency tiering (decode forwards).  The pages' engine keeps the hot
 * experts on the GPU and the rest of the expert library in host RAM ("Edge0-145B
 * en local", introduction: VRAM / RAM / SSD tiers; "Edge0-145B hardware
 * requirements", flags table: resident budget, memory-mapped experts).  Here the
 * layer's routed records live in host memory and n_slots of them are cached in
 * device memory:
 *   - each decode forward reads a resident expert from its cache slot; after its
 *     routing, the records of the chosen experts that are not resident are copied
 *     from host memory (over the host link, by all CTAs, plain loads through the
 *     device mapping) into a staging area, then the forward continues as usual;
 *   - the kernel counts how often each expert is chosen; edge0_moe_tier_rebalance
 *     moves the most-used experts into the slots (edge0_tier_plan, below).
 * The result of a forward does not depend on which experts are resident.
 *
 * edge0_moe_tier_attach: host_records = the layer's n_experts records at the
 *   handle's expert_stride, in pinned host memory mapped for device access
 *   (cudaHostAlloc / cudaMallocHost with unified addressing, or cudaHostRegister
 *   with the mapped flag), 256-byte aligned; caller-owned, valid until detach.
 *   Allocates n_slots device slots (all empty at first) and a staging area of
 *   16 * top_k records.  From then on the handle ignores desc.experts.  Requires a
 *   handle created with max_tokens <= 16 and one latent group (prefill forwards,
 *   which grouped layers run at every T, read every record from device memory:
 *   UNSUPPORTED); a second attach is UNSUPPORTED.  Synchronises.
 * edge0_moe_tier_place: puts expert slot_expert[k] (host int [n_slots], -1 =
 *   empty, no expert twice) into slot k, copying the records on `stream` and
 *   updating the table; synchronises `stream`.
 * edge0_moe_tier_rebalance: reads the use counts (synchronises `stream`), places
 *   the edge0_tier_plan choice and clears the counts.
 * edge0_moe_tier_stats: out host [4]: tiered forwards, non-resident experts
 *   copied, bytes copied from host memory, experts now resident.  Synchronises.
 * edge0_moe_tier_detach: frees the slots and staging (synchronises); the handle
 *   reads desc.experts again.
 */
edge0_status edge0_moe_tier_attach(void *handle, const void *host_records, int n_slots,
                                   edge0_stream_t stream);
edge0_status edge0_moe_tier_place(void *handle, const int *slot_expert, edge0_stream_t stream);
edge0_status edge0_moe_tier_rebalance(void *handle, edge0_stream_t stream);
edge0_status edge0_moe_tier_stats(void *handle, unsigned long long *out);
edge0_status edge0_moe_tier_detach(void *handle);

/*
 * The residency policy (host code, no device access): the n_slots experts with the
 * most uses (use host uint [n_experts]; ties to the lower index; an unused expert is
 * never promoted) are resident in `next`.  An expert already in a slot (cur host int
 * [n_slots], -1 empty) and still chosen keeps its slot; the other chosen experts fill
 * the remaining slots in rank order; a slot left over keeps its current expert.
 * Returns the number of slots whose expert changes, or -1 on bad arguments.
 * Source: hot experts resident in VRAM, the rest in host RAM ("Edge0-145B en
 * local", introduction; "Edge0-145B hardware requirements", flags table:
 * --resident-budget-gib); the most-used policy is this library's reading.
 */
int edge0_tier_plan(const unsigned int *use, int n_experts, int n_slots, const int *cur, int *next);

/*
 * Failure-path check: launch one block on `stream` that waits on an mbarrier
 * no one arrives at, through the same bounded wait every kernel of the library
 * uses (limit 1 s of %globaltimer).  The wait runs out, sets the handle's
 * error word and the block returns; the next edge0_moe_get_error on the
 * handle reports EDGE0_ERR_TIMEOUT.  Faults nothing; the handle stays usable.
 */
edge0_status edge0_moe_debug_wait_probe(void *handle, edge0_stream_t stream);

/*
 * Synchronise with the device and return the handle's device error word
 * (EDGE0_OK, or EDGE0_ERR_TIMEOUT if a bounded device wait ran out since the
 * last call); clears the word.
 */
edge0_status edge0_moe_get_error(void *handle);

/* Static text for a status code. */
const char *edge0_status_string(edge0_status status);

/* Free the handle's workspace (synchronises the device first).  NULL is a no-op. */
void edge0_moe_destroy(void *handle);

#ifdef __cplusplus
}
#endif

#endif /* EDGE0_MOE_H */
