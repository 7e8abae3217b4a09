/* coli_moe -- one int4 routed-expert MoE layer on an NVIDIA GB300 (sm_103a), C ABI.
 *
 * The layer is the MoE step of a GLM-5.2-style decoder as the colibrì pages describe it
 * ("colibrì 架构概述" §5, the moe step of each layer; §3.1 int4 experts and the IDOT integer
 * dot path; the colibrì README "絕不為同一次硬碟讀取等待兩遍" for the batch union):
 *
 *   x_n  = RMSNorm(x)                    (only with has_norm; then y = x + MoE(x_n))
 *   q8   = int8 blocks of 32 of x_n      (Q8_0-style: d = max|x|/127, q = round(x/d))
 *   route: logits = W_r x_n (fp32), score = sigmoid(logit), top-K by score + bias
 *          (bias selects only; ties go to the lower expert id), w_k = score_k / sum(score)
 *   union: the T*K (token, expert) pairs grouped by expert so each distinct expert's
 *          weights are read once per call; the shared expert (id E) takes every token
 *   expert: g = W_g x, u = W_u x (int4 weights x int8 codes, int32 block dots, per-row f32
 *          scale, per-block activation scale), h = SiLU(g) * u, h re-quantised to int8
 *          blocks of 32, e = W_d h
 *   combine: y_t = e(shared, t), then y_t = fma(w_{t,k}, e(t,k), y_t) for k = 0..K-1
 *
 * All fp32 steps follow one canonical order of operations (fma chains over 32 contiguous
 * groups, then a pairwise tree; an own exp), so results are reproducible bit for bit and a
 * token's output does not depend on the batch it is in.
 *
 * Formats.  An expert record is [gate f x d | up f x d | down d x f] int4 nibbles, row
 * major, two's complement, element 2i in the low nibble of byte i of its row, followed by
 * the f32 row scales [s_gate (f) | s_up (f) | s_down (d)] ("colibrì 架构概述" §3.1: two
 * 4-bit values per byte, one f32 scale per row; README: the three matrices of an expert
 * are stored next to each other).  A layer created with wbits = 8 takes the same record with
 * one int8 code per byte, with wbits = 2 four two's-complement 2-bit codes per byte (element
 * 4i+k in bits 2k..2k+1 of byte i of its row) (§3.1 int8 rows for the dense part and the MTP
 * head, int2 packed experimental).  The library repacks records into its own device layout
 * at load time; the weights are never expanded to floats.
 *
 * Conventions.  Every call returns COLI_OK (0) or a negative COLI_E* status; nothing aborts,
 * throws or traps.  Pointers named *_dev are device pointers owned by the caller; the
 * library owns everything it allocates in coli_moe_create and frees it in coli_moe_destroy.
 * `stream` is a cudaStream_t (NULL = legacy default stream).  Calls on one handle must not
 * overlap in time (they share its workspace).  All calls use the CUDA device that is
 * current on the calling thread; it must be the device the handle was created on.
 */
#ifndef COLI_MOE_H
#define COLI_MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define COLI_OK 0
#define COLI_EINVAL (-1)       /* bad argument (NULL pointer, size out of range, ...)      */
#define COLI_ENOMEM (-2)       /* device or host allocation failed                         */
#define COLI_ESTATE (-3)       /* call out of order (e.g. forward before weights loaded)   */
#define COLI_ECUDA (-4)        /* a CUDA runtime call or kernel launch failed              */
#define COLI_ETIMEOUT (-5)     /* a bounded device-side wait gave up (see coli_moe_status) */
#define COLI_EUNSUPPORTED (-6) /* shape the kernels do not cover (see coli_moe_create)     */
#define COLI_EIO (-7)          /* a file could not be opened, read or written in full       */

typedef struct coli_moe coli_moe; /* opaque; owned by the library */

typedef struct {
  int d;            /* model width; multiple of 128, d/32 divisible by ceil(d/1024), <= 8192  */
  int f;            /* expert hidden width (routed and shared); same rules as d              */
  int n_experts;    /* E routed experts, 1..1024                                              */
  int top_k;        /* K experts per token, 1..min(E, 32)                                      */
  int n_shared;     /* 0 or 1 always-on shared expert (id E), weight 1                        */
  int qblock;       /* activation block length; must be 32                                    */
  int max_tokens;   /* largest T accepted by forward; workspace is sized for it, 1..4096      */
  float routed_scale; /* multiplies every routing weight (1.0 = plain renormalisation)       */
  float rms_eps;    /* RMSNorm epsilon (used only with has_norm)                               */
  int has_norm;     /* 1: forward computes y = x + MoE(RMSNorm(x)) with the loaded gamma      */
  int wbits;        /* bits per expert weight: 4 (int4, also when 0), 8 (int8 rows) or 2     */
                    /* (int2 rows); int8 and int2 layers run the decode kernels for every T    */
  int hbm_slots;    /* 0 (or >= n_experts): every expert record resident in HBM.  Otherwise a   */
                    /* tiered layer: HBM holds hbm_slots routed records (>= top_k) plus the    */
                    /* shared one, every record also sits in pinned host memory, and           */
                    /* coli_tier.h's coli_moe_forward_tiered places the experts a forward needs */
} coli_moe_config;

/* Optional per-step outputs of coli_moe_forward_debug.  Device pointers owned by the caller;
 * NULL entries are skipped.  P = T*K + n_shared*T pairs, ordered as in the batch union. */
typedef struct {
  float* xn;          /* [T,d]   layer input after RMSNorm (copy of x without norm)       */
  int8_t* qx;         /* [T,d]   activation q8 codes                                      */
  float* dx;          /* [T,d/32] activation block scales                                  */
  float* logits;      /* [T,E]                                                             */
  float* scores;      /* [T,E]   sigmoid(logits)                                           */
  int32_t* ids;       /* [T,K]   selected experts, rank order                              */
  float* w;           /* [T,K]   routing weights                                           */
  int32_t* n_union;   /* [1]     union slots (distinct routed experts + shared)            */
  int32_t* union_ids; /* [E+1]   expert id per union slot, ascending, shared (= E) last     */
  int32_t* offsets;   /* [E+2]   first pair of each union slot; offsets[n_union] = P        */
  int32_t* pair_token;/* [P]     token of each pair                                        */
  int32_t* pair_rank; /* [P]     k of each pair (-1 for the shared expert)                 */
  int32_t* inv;       /* [T,K]   pair index of (t, ids[t,k])                               */
  float* g;           /* [P,f]   gate projection                                           */
  float* u;           /* [P,f]   up projection                                             */
  float* h;           /* [P,f]   SiLU(g)*u                                                 */
  int8_t* qh;         /* [P,f]   h q8 codes                                                */
  float* dh;          /* [P,f/32] h block scales                                           */
  float* e;           /* [P,d]   expert outputs                                            */
  int32_t* Ag;        /* [P,f,d/32] int32 block dots of the gate projection                */
  int32_t* Au;        /* [P,f,d/32] up                                                     */
  int32_t* Ad;        /* [P,d,f/32] down                                                   */
} coli_moe_dump;

/* Validates cfg and allocates, on the current device, the expert store ((E+n_shared) expert
 * records in the library's layout), the router and the workspace for max_tokens.  Layers with
 * d > 7168 or f > 5120 run kernel instances that spill registers (correct, slower).
 * EINVAL: bad cfg or out == NULL.  EUNSUPPORTED: a shape rule above is broken.  ENOMEM.
 * ECUDA: no usable device.  On error *out is left NULL. */
int coli_moe_create(const coli_moe_config* cfg, coli_moe** out);

/* Frees everything the handle owns (synchronises the device first).  NULL is a no-op. */
void coli_moe_destroy(coli_moe* h);

/* Copies the router W_r [E,d] (fp32, row major), the optional selection bias [E] and, for
 * has_norm, the RMSNorm gamma [d] into the handle.  Host or device pointers.  Returns when
 * the copies are complete on `stream`.  EINVAL: NULL W_r, or gamma NULL while has_norm. */
int coli_moe_load_router(coli_moe* h, const float* W_r, const float* bias, const float* gamma,
                         void* stream);

/* Loads `count` consecutive expert records, ids first..first+count-1 (id E = the shared
 * expert), from `packed` (count records of 3*d*f/2 bytes, format above) and `scales` (count
 * records of 2f+d floats).  Host or device pointers; repacked on the device.  The host
 * buffers may be freed on return (the call synchronises `stream`).  EINVAL: ids out of range. */
int coli_moe_load_experts(coli_moe* h, int first, int count, const uint8_t* packed,
                          const float* scales, void* stream);

/* y_dev[T,d] = layer(x_dev[T,d]), asynchronous on `stream`, no host synchronisation and no
 * allocation (safe to capture in a CUDA graph).  T == 0 is a no-op.  x_dev must be 16-byte
 * aligned.  x_dev may equal y_dev only with has_norm (residual update in place).  EINVAL:
 * T < 0 or T > max_tokens, NULL or misaligned pointers, forbidden aliasing.  ESTATE: router or
 * some expert not loaded yet. */
int coli_moe_forward(coli_moe* h, const float* x_dev, int T, float* y_dev, void* stream);

/* coli_moe_forward plus the intermediates selected in `dump` (slower; for verification). */
int coli_moe_forward_debug(coli_moe* h, const float* x_dev, int T, float* y_dev,
                           const coli_moe_dump* dump, void* stream);

/* coli_moe_forward that also records `events[0..3]` (cudaEvent_t handles created by the
 * caller) on `stream`: before the routing kernel(s), after them, after the gate/up kernel and
 * after the down kernel -- so the caller can time each launch.  When the forward runs the expert
 * half as one fused kernel (coli_moe_launches returns 2) events 1..2 bracket that kernel and
 * events 2..3 nothing; on the batched tensor-core path events 0..1 bracket the five routing
 * launches and events 2..3 the down GEMM and the combine.  The events serialise the launches (no
 * programmatic overlap between them).  T <= 4, or a batch that takes the tensor-core path.
 * EINVAL: n_events < 4 or T out of range. */
int coli_moe_forward_profiled(coli_moe* h, const float* x_dev, int T, float* y_dev,
                              void* const* events, int n_events, void* stream);

/* Host-buffer form: copies x_host [T,d] to the device, runs forward, copies y back to
 * y_host [T,d] and returns once y_host holds the result; any host memory (pageable or pinned).
 * Batches of up to 8 tokens go through the handle's own mapped pinned staging and one CUDA graph
 * per token count (a kernel that reads x from the staging, the forward's kernels, a kernel that
 * writes y and the status word back and then raises a completion counter in the staging),
 * captured on the handle's stream on the first call with that count and launched on `stream`;
 * the call waits by polling that counter (falling back to synchronising `stream` after a
 * second), so on return the graph's last kernel may still be exiting on `stream` -- later work
 * on `stream` is ordered after it as usual, and other streams must synchronise with `stream`
 * before relying on the call's device-side effects.  Larger batches, and tiered layers, copy
 * directly and synchronise `stream`.  Returns COLI_ETIMEOUT (and clears it, as coli_moe_status
 * does) when a bounded device wait of this forward gave up; y_host is then undefined. */
int coli_moe_forward_host(coli_moe* h, const float* x_host, int T, float* y_host, void* stream);

/* Runs n_layers has_norm layers in sequence on x_dev [T,d] in place:
 * x <- x + MoE_l(RMSNorm_l(x)) for l = 0..n_layers-1.  Asynchronous on `stream`. */
int coli_moe_stack_forward(coli_moe* const* layers, int n_layers, float* x_dev, int T,
                           void* stream);

/* Device status word of the handle: COLI_OK, or COLI_ETIMEOUT if a bounded device-side wait
 * of an earlier forward gave up (the word is then cleared).  Synchronises `stream`. */
int coli_moe_status(coli_moe* h, void* stream);

/* Batches of at least min_tokens tokens (min_tokens >= 2) take the batched tensor-core path
 * (when the handle has it: max_tokens > 8); smaller batches run the decode kernels, in one union
 * pass of up to 8 tokens or in chunks of 8.  Both give the same result for every token.  The
 * default, 128, is where the two cost about the same on the GLM-shaped layer.  EINVAL:
 * min_tokens < 2. */
int coli_moe_set_prefill_min(coli_moe* h, int min_tokens);

/* Failure-path test knob.  fault = COLI_FAULT_SKIP_ARRIVAL makes the next one-token forward on
 * this handle that runs the fused expert kernel (coli_moe_launches(h, 1) == 2) leave CTA 0 out
 * of that kernel's grid barrier: every CTA's bounded wait at the barrier then runs out (about
 * 2 s), the call's output is undefined and coli_moe_status reports COLI_ETIMEOUT; nothing
 * hangs and the handle stays usable.  The knob applies to one such forward and then clears
 * itself; fault = 0 clears it.  Not for production use (and not to be captured in a CUDA
 * graph: the knob is read when the forward is launched).  EINVAL: unknown fault code. */
#define COLI_FAULT_SKIP_ARRIVAL 1
int coli_moe_inject_fault(coli_moe* h, int fault);

/* Number of kernel launches one coli_moe_forward of T tokens makes on this handle: 2 for one
 * token when the expert half runs as one fused kernel (router, then gate/up + down), 3 per
 * chunk of at most 8 tokens on the decode path (router, gate/up, down; one union pass per
 * chunk), 8 on the batched tensor-core path (batches of at least the coli_moe_set_prefill_min
 * size, 128 by default).  Negative status on error (EINVAL: T < 1 or T > max_tokens). */
int coli_moe_launches(const coli_moe* h, int T);

/* Bytes of one expert record in the canonical format (3*d*f/2 + 4*(2f+d)). */
int64_t coli_moe_expert_record_bytes(int d, int f);

/* The same for wbits = 4, 8 or 2 bits per weight (3*d*f*wbits/8 + 4*(2f+d)); EINVAL for
 * another width. */
int64_t coli_moe_expert_record_bytes_w(int d, int f, int wbits);

/* Standalone pack of fp32 rows into the canonical int4 format ("colibrì 架构概述" §3.1):
 * s[r] = max|w[r,:]|/7, q = round(w/s) clamped to [-7,7], two nibbles per byte.
 * w_dev [rows,cols] -> packed_dev [rows,cols/2], scales_dev [rows].  cols even, <= 65536. */
int coli_quantize_i4_rows(const float* w_dev, int64_t rows, int cols, uint8_t* packed_dev,
                          float* scales_dev, void* stream);

/* Standalone pack of fp32 rows into int8 rows ("colibrì 架构概述" §3.1 int8, quantize_rows):
 * s[r] = max|w[r,:]|/127, q = round(w/s) (half away from zero) clamped to [-127,127], one code
 * per byte.  w_dev [rows,cols] -> q_dev [rows,cols], scales_dev [rows].  cols <= 65536. */
int coli_quantize_i8_rows(const float* w_dev, int64_t rows, int cols, int8_t* q_dev,
                          float* scales_dev, void* stream);

/* Standalone pack of fp32 rows into int2 rows ("colibrì 架构概述" §3.1 int2 packed, pack_int2):
 * s[r] = max|w[r,:]|, q = round(w/s) clamped to [-1,1], four two's-complement 2-bit codes per
 * byte, element 4i+k in bits 2k..2k+1 of byte i.  w_dev [rows,cols] (16-byte aligned) ->
 * packed_dev [rows,cols/4], scales_dev [rows].  cols a multiple of 4, <= 65536. */
int coli_quantize_i2_rows(const float* w_dev, int64_t rows, int cols, uint8_t* packed_dev,
                          float* scales_dev, void* stream);

/* Standalone Q8_0-style activation quantisation: blocks of 32, d = max|x|/127,
 * q = round(x/d).  x_dev [n] -> q_dev [n], d_dev [n/32]; n a multiple of 32. */
int coli_quantize_act_q8(const float* x_dev, int64_t n, int8_t* q_dev, float* d_dev,
                         void* stream);

/* Routing without allocating anything: the layer's router alone (fp32 logits, sigmoid, top-K by
 * score + optional selection bias with ties to the lower id, weights renormalised over the
 * selected scores) -- bit-identical to the ids and weights coli_moe_forward uses for the same
 * inputs (without RMSNorm).  The source pages have no counterpart: this is an interface for
 * callers that cannot call cudaMalloc, such as a process whose device memory is owned entirely
 * by another allocator (a serving framework that reserves the device up front and hands out
 * pieces of its own pool), where a direct allocation would fail or break that allocator's
 * accounting.  It needs no handle: x_dev [T,d], W_r_dev [E,d] (row major), bias_dev [E] or
 * NULL, outputs ids_dev [T,K] and w_dev [T,K], all device pointers owned by the caller; x_dev
 * and W_r_dev 16-byte aligned.  Limits: T <= 4, T*E <= 4096, E <= 1024, K <= min(E, 32), d a
 * multiple of 128 up to 8192 (EINVAL beyond them).  Its scratch (16 KB) is a fixed array in the
 * library's device memory, present on every device that loads the library until the process
 * exits; the first call on a device looks up that array's address and keeps it (make that first
 * call before any stream capture), so calls after a cudaDeviceReset of that device are not
 * supported.  Every call shares the array: calls that overlap on the GPU (for example on two
 * streams) race on it. */
int coli_route_noalloc(const float* x_dev, int T, const float* W_r_dev, const float* bias_dev,
                       int E, int d, int K, float routed_scale, int32_t* ids_dev, float* w_dev,
                       void* stream);

const char* coli_moe_strerror(int status);

#ifdef __cplusplus
}
#endif
#endif /* COLI_MOE_H */
