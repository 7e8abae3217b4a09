// Internal types of the coli_moe library: device layout of the expert store, the per-handle
// workspace and the kernel launchers.  Not part of the C ABI.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "coli_moe.h"

namespace coli {

constexpr int kQB = 32;                         // activation block length
constexpr int kDecodeTmax = 8;                  // tokens per call on the smem-staged path
constexpr int kRouteTgroup = 4;                 // tokens the router stages at a time
constexpr int kNW = 8;                          // consumer warps per CTA of the expert kernels
constexpr int kThreads = (kNW + 1) * 32;        // + one producer warp
constexpr int kGuRps = 8;                       // gate/up row pairs per pipeline stage
constexpr int kDownRowsPerWarp = 8;             // output rows per warp per down stage
constexpr int kDownChunk = kNW * kDownRowsPerWarp;  // at most this many rows per down stage
constexpr int kMaxStages = 8;
// Default batch size from which the tensor-core path is taken: below it the decode kernels in
// chunks of 4 tokens are faster (measured on the GLM layer: 188 vs 1178 us at 5 tokens, 4.4 vs
// 8.4 ms at 128, even at 256, 17.5 vs 9.1 ms at 512)
constexpr int kPrefillMinTokens = 128;
constexpr int kSmemLimit = 232448 - 1024;       // 227 KB per CTA minus room for static smem
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // bounded device waits give up after 2 s
constexpr int kPrefillTileN = 32;               // pairs per tensor-core tile

// Store layout (built by the repack kernel at load time):
//  * a matrix row of n int4 values is n/32 blocks of 16 bytes.  With nb = n/32 blocks and
//    G = ceil(nb/32) blocks per lane group, block b = g*G + i is stored at chunk position
//    g*G + ((i + ((g>>2)&1)) mod G): each group's blocks stay contiguous (a K-range a matrix
//    engine can load whole) and the rotation keeps a warp's loads free of bank conflicts.
//    Inside a chunk, word k holds elements 8k..8k+7: byte m has element 8k+m in the low
//    nibble and 8k+m+4 in the high nibble, each as code + 8 (0..15).
//  * wgu: per expert slot, f rows of [gate row r | up row r] (d bytes per row pair).
//  * wd : per expert slot, d rows of the down matrix (f/2 bytes each).
//  * sc : per expert slot, the canonical scales [s_gate f | s_up f | s_down d].
//  * wr : router rows with 4-float chunks permuted the same way (lane g's 4*i..4*i+3 of its
//    d/32 contiguous elements at chunk i*32 + g).
struct Store {
  uint8_t* wgu = nullptr;
  uint8_t* wd = nullptr;
  float* sc = nullptr;
  float* wr = nullptr;
  float* bias = nullptr;   // nullptr: no selection bias
  float* gamma = nullptr;  // has_norm only
  // tiered layers (fewer HBM slots than experts): the store slot of each expert id, -1 when not
  // resident; nullptr: every expert sits in the slot of its own id
  const int32_t* slot_of = nullptr;
};

struct Work {
  float* xn = nullptr;       // [Tm,d]  normalised input (natural layout)
  float* xnp = nullptr;      // [Tm,d]  same, router chunk layout
  int8_t* qx = nullptr;      // [Tm,d]
  float* dx = nullptr;       // [Tm,d/32]
  int32_t* sx = nullptr;     // [Tm,d/32] sum of the codes of each block
  float* logits = nullptr;   // [Tm,E]
  float* scores = nullptr;   // [Tm,E]
  int32_t* ids = nullptr;    // [Tm,K]
  float* w = nullptr;        // [Tm,K]
  int32_t* n_union = nullptr;
  int32_t* union_ids = nullptr;  // [E+1]
  int32_t* offsets = nullptr;    // [E+2]
  int32_t* pair_token = nullptr; // [Pm]
  int32_t* pair_rank = nullptr;  // [Pm]
  int32_t* inv = nullptr;        // [Tm,K]
  float* hf = nullptr;       // [Pm,f]  SwiGLU output h (fp32) before re-quantisation
  int8_t* qh = nullptr;      // [Pm,f]
  float* dh = nullptr;       // [Pm,f/32]
  int32_t* sh = nullptr;     // [Pm,f/32]
  int32_t* sel_flag = nullptr;  // [0] 1 once the gate/up grid of the current call published its
                                // expert selection; [1] the fused kernel's barrier counter
                                // (the router grid clears both)
  int32_t* status = nullptr;   // COLI_OK or COLI_ETIMEOUT
};

// workspace of the batched (tensor-core) path; rows padded by one tile for the copies
struct PrefillWork {
  __nv_bfloat16* xb = nullptr;  // [Pm+64][d] every pair's activation codes as bf16
  float* dxp = nullptr;         // [Pm+64][d/32] their block scales
  __nv_bfloat16* hb = nullptr;  // [Pm+64][f] h codes as bf16 (down projection operand)
  float* e = nullptr;           // [Pm][d] expert outputs per pair
  int32_t* tile_prefix = nullptr;  // [E+2] per union slot: tiles of kPrefillTileN pairs before it
};

struct PrefillMaps {
  CUtensorMap wgu, wd, xb, hb, wr, xnp;
};

struct Shape {
  int d, f, E, K, n_shared, T;
  float routed_scale, rms_eps;
  int has_norm;
  int wbits;  // bits per expert weight: 4, 8 or 2
};

// optional debug outputs of the expert kernels (device pointers, may be null)
struct ExpertDebug {
  float* g = nullptr;
  float* u = nullptr;
  float* e = nullptr;
  int32_t* Ag = nullptr;
  int32_t* Au = nullptr;
  int32_t* Ad = nullptr;
};

// ---- launchers (return the launch's cudaError_t) ----
// `pdl`: launch as a programmatic dependent of the previous kernel in the stream (the kernel
// prefetches weights before waiting for its predecessor's results)
cudaError_t launch_route(const float* x, const Shape& s, const Store& st, const Work& w,
                         cudaStream_t stream);
cudaError_t launch_gateup_decode(const Shape& s, const Store& st, const Work& w,
                                 const ExpertDebug& dbg, int num_sms, bool pdl,
                                 cudaStream_t stream);
cudaError_t launch_down_decode(const float* x, float* y, const Shape& s, const Store& st,
                               const Work& w, const ExpertDebug& dbg, int num_sms, bool pdl,
                               cudaStream_t stream);
cudaError_t configure_route_kernels();
cudaError_t launch_select_publish(const Shape& s, const Store& st, const Work& w,
                                  cudaStream_t stream);
// up to kSlotUpdateMax slot-table entries of a tiered layer, passed by value to one launch
constexpr int kSlotUpdateMax = 64;
struct SlotUpdate {
  int n;
  int32_t ids[kSlotUpdateMax];
  int32_t slots[kSlotUpdateMax];
};
cudaError_t launch_set_slots(int32_t* slot_of, const SlotUpdate& u, cudaStream_t stream);
cudaError_t configure_route_batch_kernels(int E);
cudaError_t launch_route_batch(const float* x, const Shape& s, const Store& st, const Work& w,
                               const CUtensorMap& map_wr, const CUtensorMap& map_x,
                               int32_t* tile_prefix, int tile_n, __nv_bfloat16* xb, float* dxp,
                               cudaStream_t stream);
cudaError_t configure_prefill_kernels(int d, int f, int E);
int prefill_smem_bytes(int d, int f, int E, int down);
bool prefill_make_maps(PrefillMaps* maps, const Store& st, const Work& w, const PrefillWork& pw,
                       int d, int f, int E, int slots, int prow, int tmax);
cudaError_t launch_prefill_experts(const float* x, float* y, const Shape& s, const Store& st,
                                   const Work& w, const PrefillWork& pw, const PrefillMaps& maps,
                                   const ExpertDebug& dbg, int num_sms, cudaStream_t stream,
                                   cudaEvent_t after_gateup = nullptr);
cudaError_t launch_repack_matrix(const uint8_t* src, uint8_t* dst, int rows, int cols,
                                 int64_t dst_row_stride, cudaStream_t stream, int wbits);
cudaError_t launch_quantize_i8_rows(const float* w, int64_t rows, int cols, int8_t* q,
                                    float* scales, cudaStream_t stream);
cudaError_t launch_quantize_i2_rows(const float* w, int64_t rows, int cols, uint8_t* packed,
                                    float* scales, cudaStream_t stream);
cudaError_t launch_permute_router(const float* src, float* dst, int E, int d,
                                  cudaStream_t stream);
cudaError_t launch_quantize_i4_rows(const float* w, int64_t rows, int cols, uint8_t* packed,
                                    float* scales, cudaStream_t stream);
cudaError_t launch_quantize_q8(const float* x, int64_t n, int8_t* q, float* d,
                               cudaStream_t stream);
// host-buffer forwards: n floats (a multiple of 4) from / to mapped pinned host memory
// the host-buffer forward's staging tail: word 0 = the status word, word kHostDoneWord = a
// completion counter the last kernel of each call raises by one
constexpr int kHostDoneWord = 4;
cudaError_t launch_host_in(const float* hx, float* dx, int n, cudaStream_t stream);
cudaError_t launch_host_out(const float* dy, float* hy, int n, const int* status, int* hstatus,
                            cudaStream_t stream);
cudaError_t configure_expert_kernels();

// per-CTA unit table of the gate/up kernel: slot, expert, first pair, pair count, the pairs'
// tokens (T at most) and the 32 gate + 32 up row scales
constexpr int kGuTabInts = 5 + kDecodeTmax;  // slot, expert, first pair, pairs, hb, tokens
constexpr int kGuTabBytes = (kGuTabInts + 64) * 4;
// Relative cost of one gate/up unit whose union slot serves np tokens: its bytes take the same
// time whatever np (kGuCostBytes), its dots grow with np (kGuCostPair each); the larger bounds
// the unit.  The routed units are split over the CTAs by this cost, not by count.  Calibrated
// on the four-token int4 GLM layer: a four-token unit measured about 3.6 times a one-token unit,
// and the step time keeps improving up to a model ratio of about 4.4, flat beyond.
constexpr int kGuCostBytes = 20, kGuCostPair = 22;
__host__ __device__ constexpr int gu_unit_cost(int np) {
  return kGuCostPair * np > kGuCostBytes ? kGuCostPair * np : kGuCostBytes;
}

// Gate/up row pairs per ring stage: 8 (one per consumer warp, each warp reduces the gate and the
// up row of its pair) for int4 and int2; 4 for int8, whose rows are twice the int4 bytes: warp w
// then reduces one row, the gate row of pair w%4 (w < 4) or its up row, and SwiGLU is applied
// when the unit's 32 rows are in.
__host__ __device__ constexpr int gu_rows_per_stage(int wb) { return wb == 8 ? 4 : 8; }
// Down rows per stage chunk: at most 8 per warp, and half that for int8 so that a stage keeps the
// bytes of an int4 one.
__host__ __device__ constexpr int dn_chunk_cap(int wb) { return wb == 8 ? kDownChunk / 2 : kDownChunk; }

// shared-memory plans (host and device agree on the carve-up)
struct GateupPlan {
  int nst, stage_bytes, xs_bytes, aux_bytes, hs_bytes, tab_bytes, sel_bytes, max_units, total;
};
// down kernel: a stage holds one chunk of a union expert's down rows, then the h codes, block
// scales and code sums of that expert's pairs (at most T of them)
struct DownPlan {
  int nst, stage_bytes, w_bytes, es_bytes, tab_bytes, sel_bytes, max_rows, max_slots, total;
};
// shared-memory plan of the fused one-token expert kernel (gate/up ring, a region used first by
// the gate/up phase and then by the down phase, the selection)
struct FusedPlan {
  int nst, stage_bytes, xs_bytes, aux_bytes, hs_bytes, tab_bytes, max_units;
  int hq_bytes, haux_bytes, es_bytes, tsd_bytes, max_rows, chunk, max_slots;
  int region, sel_bytes, total;
};
FusedPlan fused_plan(int d, int f, int K, int E, int n_shared, int grid);
bool fused_supported(int d, int f, int K, int E, int n_shared, int num_sms);
cudaError_t configure_fused_kernels();
cudaError_t launch_expert_fused(const float* x, float* y, const Shape& s, const Store& st,
                                const Work& w, const ExpertDebug& dbg, int num_sms, bool pdl,
                                bool skip_arrival, cudaStream_t stream);
GateupPlan gateup_plan(int d, int f, int T, int K, int E, int n_shared, int grid, int wbits);
DownPlan down_plan(int d, int f, int T, int K, int E, int n_shared, int grid, int wbits);
int down_grid(int d, int num_sms);  // CTAs of the down kernel
// the decode kernels of one weight width (expert_decode.cuh, instantiated per width)
template <int WB> cudaError_t configure_gateup_kernels_wb();
template <int WB> cudaError_t configure_down_kernels_wb();
template <int WB>
cudaError_t launch_gateup_decode_wb(const Shape& s, const Store& st, const Work& w,
                                    const ExpertDebug& dbg, int num_sms, bool pdl,
                                    cudaStream_t stream);
template <int WB>
cudaError_t launch_down_decode_wb(const float* x, float* y, const Shape& s, const Store& st,
                                  const Work& w, const ExpertDebug& dbg, int num_sms, bool pdl,
                                  cudaStream_t stream);

}  // namespace coli
