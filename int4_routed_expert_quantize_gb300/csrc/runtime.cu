// Host runtime of the coli_moe C ABI: argument checks, allocation of the expert store and
// workspace, weight loading (with the repack into the store layout) and the launch sequence
// of one forward: prep -> router (+ top-K, union) -> gate/up SwiGLU -> down + combine.
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include <chrono>
#include <cmath>
#include <mutex>
#include <new>
#include <vector>

#include "coli_internal.h"
#include "coli_moe.h"
#include "coli_tier.h"

using namespace coli;

namespace {
constexpr int kHostGraphMaxT = 8;  // token counts whose host-buffer forward runs as a cached graph
}

struct coli_moe {
  coli_moe_config cfg{};
  int device = 0;
  int num_sms = 0;
  int slots = 0;  // E + n_shared
  Store st;
  Work w;
  float* dev_io = nullptr;  // [2][Tm][d] buffers of coli_moe_forward_host
  // coli_moe_forward_host for small batches: pinned staging for x, y and the status word, and
  // one instantiated graph per token count (copy in, the forward's kernels, copy out, status)
  float* pin_x = nullptr;          // host addresses
  float* pin_y = nullptr;
  int32_t* pin_status = nullptr;    // [0] status word, [kHostDoneWord] completion counter
  int32_t host_done = 0;             // the counter's value after the last completed call
  float* map_x = nullptr;          // the same memory as the device addresses it
  float* map_y = nullptr;
  int32_t* map_status = nullptr;
  cudaStream_t cap_stream = nullptr;
  cudaGraphExec_t host_graph[kHostGraphMaxT + 1] = {};
  bool prefill = false;     // the tensor-core path is set up (max_tokens > kDecodeTmax)
  int prefill_min = kPrefillMinTokens;  // batches of at least this many tokens take it
  bool fused = false;       // one-token forwards use the fused expert kernel
  int decode_tmax = 1;      // tokens per launch of the decode kernels (<= kDecodeTmax)
  int fault = 0;            // one-shot failure-path knob (coli_moe_inject_fault)
  PrefillWork pw;
  PrefillMaps maps;
  bool router_loaded = false;
  std::vector<uint8_t> loaded;
  int n_loaded = 0;
  std::vector<void*> allocs;
  // Tiered layer (0 < hbm_slots < E): HBM holds hbm_slots routed records and, in the slot after
  // them, the shared one; every record also sits in pinned host memory in the store layout,
  // from where the placements copy it.  The kernels address records through the device slot
  // table; slot_owner mirrors it on the host.
  int hbm_slots = 0;  // 0: every expert resident in the slot of its own id
  uint8_t* host_wgu = nullptr;
  uint8_t* host_wd = nullptr;
  float* host_sc = nullptr;
  int32_t* slot_of = nullptr;         // device [E+1]
  std::vector<int32_t> slot_owner;    // expert in each device slot (-1: free)
  int32_t* pin_union = nullptr;       // pinned [E+2]: n_union, then the union's expert ids
  cudaEvent_t copy_done = nullptr;    // after the last placement made outside a forward
  cudaEvent_t fwd_done = nullptr;     // after the last forward's kernels
  bool copy_pending = false;          // a forward must wait for copy_done first
  int64_t copied_records = 0, copied_bytes = 0;
  std::vector<void*> host_allocs;
};

namespace {

// bytes of the codes of one expert record: gate, up and down at wb bits per weight
int64_t rec_bytes(int d, int f, int wb) { return 3LL * d * f * wb / 8; }

bool shape_ok(int n) {
  if (n < 128 || n > 8192 || n % 128) return false;
  const int nb = n / 32, G = (nb + 31) / 32;
  return nb % G == 0;
}

int cuda_status(cudaError_t e) { return e == cudaSuccess ? COLI_OK : COLI_ECUDA; }

template <class T>
int dalloc(coli_moe* h, T** p, size_t bytes) {
  *p = nullptr;
  if (bytes == 0) bytes = 16;
  void* q = nullptr;
  if (cudaMalloc(&q, bytes) != cudaSuccess) {
    cudaGetLastError();
    return COLI_ENOMEM;
  }
  h->allocs.push_back(q);
  *p = static_cast<T*>(q);
  return COLI_OK;
}

void drop_host_graphs(coli_moe* h) {
  bool any = false;
  for (cudaGraphExec_t g : h->host_graph) any = any || g;
  if (any) cudaDeviceSynchronize();  // a call may still be finishing its last kernel
  for (cudaGraphExec_t& g : h->host_graph)
    if (g) {
      cudaGraphExecDestroy(g);
      g = nullptr;
    }
}

void free_all(coli_moe* h) {
  drop_host_graphs(h);
  for (void* p : h->host_allocs) cudaFreeHost(p);
  h->host_allocs.clear();
  if (h->copy_done) cudaEventDestroy(h->copy_done);
  if (h->fwd_done) cudaEventDestroy(h->fwd_done);
  h->copy_done = h->fwd_done = nullptr;
  if (h->cap_stream) cudaStreamDestroy(h->cap_stream);
  h->cap_stream = nullptr;
  if (h->pin_x) cudaFreeHost(h->pin_x);
  h->pin_x = h->pin_y = nullptr;
  h->pin_status = nullptr;
  for (void* p : h->allocs) cudaFree(p);
  h->allocs.clear();
}

bool is_device_ptr(const void* p) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged;
}

bool overlap(const void* a, size_t na, const void* b, size_t nb) {
  const char *pa = (const char*)a, *pb = (const char*)b;
  return pa < pb + nb && pb < pa + na;
}

int check_device(const coli_moe* h) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return COLI_ECUDA;
  return dev == h->device ? COLI_OK : COLI_ESTATE;
}

// batches of at least prefill_min tokens (>= 2) take the tensor-core path when the handle has it
bool takes_batched(const coli_moe* h, int T) {
  return h->prefill && T >= 2 && T >= h->prefill_min;
}

Shape shape_of(const coli_moe* h, int T) {
  const coli_moe_config& c = h->cfg;
  return Shape{c.d, c.f, c.n_experts, c.top_k, c.n_shared, T, c.routed_scale, c.rms_eps,
               c.has_norm, c.wbits};
}

int copy_dump(coli_moe* h, int T, const coli_moe_dump* dump, cudaStream_t stream);

// The kernels' shared-memory attributes are set per device (cudaFuncSetAttribute applies to the
// current device's context), once for each device a handle is created on.
constexpr int kMaxDevices = 64;
bool g_configured[kMaxDevices] = {};
std::mutex g_cfg_mutex;

cudaError_t configure_device(int dev) {
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_cfg_mutex);
  if (g_configured[dev]) return cudaSuccess;
  cudaError_t e = configure_expert_kernels();
  if (e == cudaSuccess) e = configure_route_kernels();
  if (e == cudaSuccess) e = configure_fused_kernels();
  if (e == cudaSuccess) g_configured[dev] = true;
  return e;
}

int run_decode(coli_moe* h, const float* x, int T, float* y, const coli_moe_dump* dump,
               cudaStream_t stream, cudaEvent_t const* ev = nullptr) {
  const Shape s = shape_of(h, T);
  ExpertDebug dbg;
  if (dump) {
    dbg.g = dump->g;
    dbg.u = dump->u;
    dbg.e = dump->e;
    dbg.Ag = dump->Ag;
    dbg.Au = dump->Au;
    dbg.Ad = dump->Ad;
    if ((dbg.g || dbg.u) && !(dbg.g && dbg.u)) return COLI_EINVAL;
    if ((dbg.Ag || dbg.Au) && !(dbg.Ag && dbg.Au)) return COLI_EINVAL;
  }
  // route -> gate/up -> down, or for one token route -> the fused expert kernel; every launch
  // after the first is a programmatic dependent that prefetches weights before waiting (the
  // router itself waits for the preceding grid before it reads anything), unless events are recorded between the launches (with the fused kernel the
  // events bracket route | fused | nothing)
  const bool pdl = (ev == nullptr);
  cudaError_t e = ev ? cudaEventRecord(ev[0], stream) : cudaSuccess;
  if (e == cudaSuccess) e = launch_route(x, s, h->st, h->w, stream);
  if (e == cudaSuccess && ev) e = cudaEventRecord(ev[1], stream);
  if (T == 1 && h->fused) {
    if (e == cudaSuccess)
      e = launch_expert_fused(x, y, s, h->st, h->w, dbg, h->num_sms, pdl,
                              h->fault == COLI_FAULT_SKIP_ARRIVAL, stream);
    h->fault = 0;
    if (e == cudaSuccess && ev) e = cudaEventRecord(ev[2], stream);
  } else {
    if (e == cudaSuccess) e = launch_gateup_decode(s, h->st, h->w, dbg, h->num_sms, pdl, stream);
    if (e == cudaSuccess && ev) e = cudaEventRecord(ev[2], stream);
    if (e == cudaSuccess) e = launch_down_decode(x, y, s, h->st, h->w, dbg, h->num_sms, pdl, stream);
  }
  if (e == cudaSuccess && ev) e = cudaEventRecord(ev[3], stream);
  if (e != cudaSuccess) return COLI_ECUDA;
  return dump ? copy_dump(h, T, dump, stream) : COLI_OK;
}

int run_prefill(coli_moe* h, const float* x, int T, float* y, const coli_moe_dump* dump,
                cudaStream_t stream, cudaEvent_t const* ev = nullptr) {
  const Shape s = shape_of(h, T);
  ExpertDebug dbg;
  if (dump) {
    dbg.g = dump->g;
    dbg.u = dump->u;
    dbg.Ag = dump->Ag;
    dbg.Au = dump->Au;
    dbg.Ad = dump->Ad;
    if ((dbg.g || dbg.u) && !(dbg.g && dbg.u)) return COLI_EINVAL;
    if ((dbg.Ag || dbg.Au) && !(dbg.Ag && dbg.Au)) return COLI_EINVAL;
  }
  cudaError_t e = ev ? cudaEventRecord(ev[0], stream) : cudaSuccess;
  if (e == cudaSuccess)
    e = launch_route_batch(x, s, h->st, h->w, h->maps.wr, h->maps.xnp, h->pw.tile_prefix,
                           kPrefillTileN, h->pw.xb, h->pw.dxp, stream);
  if (e == cudaSuccess && ev) e = cudaEventRecord(ev[1], stream);
  if (e == cudaSuccess)
    e = launch_prefill_experts(x, y, s, h->st, h->w, h->pw, h->maps, dbg, h->num_sms, stream,
                               ev ? ev[2] : nullptr);
  if (e == cudaSuccess && ev) e = cudaEventRecord(ev[3], stream);
  if (e != cudaSuccess) return COLI_ECUDA;
  if (dump) {
    const long P = (long)T * h->cfg.top_k + (h->cfg.n_shared ? T : 0);
    if (dump->e && cudaMemcpyAsync(dump->e, h->pw.e, sizeof(float) * P * h->cfg.d,
                                   cudaMemcpyDeviceToDevice, stream) != cudaSuccess)
      return COLI_ECUDA;
    return copy_dump(h, T, dump, stream);
  }
  return COLI_OK;
}

int copy_dump(coli_moe* h, int T, const coli_moe_dump* dump, cudaStream_t stream) {
  {
    const coli_moe_config& c = h->cfg;
    const long P = (long)T * c.top_k + (c.n_shared ? T : 0);
    struct Cp {
      void* dst;
      const void* src;
      size_t bytes;
    } cps[] = {
        {dump->xn, h->w.xn, sizeof(float) * T * c.d},
        {dump->qx, h->w.qx, (size_t)T * c.d},
        {dump->dx, h->w.dx, sizeof(float) * T * (c.d / 32)},
        {dump->logits, h->w.logits, sizeof(float) * T * c.n_experts},
        {dump->scores, h->w.scores, sizeof(float) * T * c.n_experts},
        {dump->ids, h->w.ids, sizeof(int32_t) * T * c.top_k},
        {dump->w, h->w.w, sizeof(float) * T * c.top_k},
        {dump->n_union, h->w.n_union, sizeof(int32_t)},
        {dump->union_ids, h->w.union_ids, sizeof(int32_t) * (c.n_experts + 1)},
        {dump->offsets, h->w.offsets, sizeof(int32_t) * (c.n_experts + 2)},
        {dump->pair_token, h->w.pair_token, sizeof(int32_t) * P},
        {dump->pair_rank, h->w.pair_rank, sizeof(int32_t) * P},
        {dump->inv, h->w.inv, sizeof(int32_t) * T * c.top_k},
        {dump->h, h->w.hf, sizeof(float) * P * c.f},
        {dump->qh, h->w.qh, (size_t)P * c.f},
        {dump->dh, h->w.dh, sizeof(float) * P * (c.f / 32)},
    };
    for (const Cp& cp : cps)
      if (cp.dst && cudaMemcpyAsync(cp.dst, cp.src, cp.bytes, cudaMemcpyDeviceToDevice, stream) !=
                        cudaSuccess)
        return COLI_ECUDA;
  }
  return COLI_OK;
}

int forward_impl(coli_moe* h, const float* x, int T, float* y, const coli_moe_dump* dump,
                 void* stream) {
  if (!h || T < 0 || T > h->cfg.max_tokens) return COLI_EINVAL;
  if (T == 0) return COLI_OK;
  if (!x || !y || ((uintptr_t)x & 15u) || ((uintptr_t)y & 3u)) return COLI_EINVAL;
  const size_t bytes = sizeof(float) * (size_t)T * h->cfg.d;
  if (x != y && overlap(x, bytes, y, bytes)) return COLI_EINVAL;
  if (x == y && !h->cfg.has_norm) return COLI_EINVAL;
  const bool batched = takes_batched(h, T);
  if (dump && T > h->decode_tmax && !batched) return COLI_EUNSUPPORTED;
  if (!h->router_loaded || h->n_loaded < h->slots) return COLI_ESTATE;
  int rc = check_device(h);
  if (rc) return rc;
  cudaStream_t st = (cudaStream_t)stream;
  if (h->hbm_slots && h->copy_pending) {  // placements made outside a forward land first
    if (cudaStreamWaitEvent(st, h->copy_done, 0) != cudaSuccess) return COLI_ECUDA;
    h->copy_pending = false;
  }
  if (batched) return run_prefill(h, x, T, y, dump, st);
  // the smem-staged kernels take up to decode_tmax tokens; larger batches run in chunks,
  // which gives the same result per token (each token's output depends on itself only)
  const int tm = h->decode_tmax;
  for (int c0 = 0; c0 < T; c0 += tm) {
    const int Tc = T - c0 < tm ? T - c0 : tm;
    rc = run_decode(h, x + (size_t)c0 * h->cfg.d, Tc, y + (size_t)c0 * h->cfg.d, dump, st);
    if (rc) return rc;
  }
  if (h->hbm_slots && cudaEventRecord(h->fwd_done, st) != cudaSuccess) return COLI_ECUDA;
  return COLI_OK;
}

// Carries out a placement decided by the tier manager on stream `st`: the evicted (or dropped)
// experts leave the slot table; each fetched record is copied from its pinned host copy into
// its HBM slot (gate/up rows, down rows, scales: one copy each) and enters the slot table.  The
// table changes follow the copies in stream order, in launches of up to kSlotUpdateMax entries.
int place(coli_moe* h, const int32_t* out_ids, const int32_t* out_slots, int n_out,
          const int32_t* in_ids, const int32_t* in_slots, int n_in, cudaStream_t st) {
  const size_t d = h->cfg.d, f = h->cfg.f, wb = h->cfg.wbits;
  const size_t gu = f * (2 * d * wb / 8), dn = d * (f * wb / 8), scn = 2 * f + d;
  SlotUpdate u{};
  bool ok = true;
  auto flush = [&]() {
    if (ok && u.n) ok = launch_set_slots(h->slot_of, u, st) == cudaSuccess;
    u.n = 0;
  };
  auto add = [&](int32_t id, int32_t slot) {
    if (u.n == kSlotUpdateMax) flush();
    u.ids[u.n] = id;
    u.slots[u.n] = slot;
    ++u.n;
  };
  for (int i = 0; i < n_out; ++i) {
    const int32_t sl = out_slots[i];
    if (sl < 0 || sl >= h->hbm_slots || h->slot_owner[sl] != out_ids[i]) return COLI_ESTATE;
    h->slot_owner[sl] = -1;
    add(out_ids[i], -1);
  }
  for (int i = 0; i < n_in && ok; ++i) {
    const int32_t id = in_ids[i], sl = in_slots[i];
    if (id < 0 || id >= h->cfg.n_experts || sl < 0 || sl >= h->hbm_slots) return COLI_ESTATE;
    if (h->slot_owner[sl] >= 0) add(h->slot_owner[sl], -1);  // not expected: the tier frees first
    ok = cudaMemcpyAsync(h->st.wgu + sl * gu, h->host_wgu + id * gu, gu, cudaMemcpyHostToDevice, st) == cudaSuccess &&
         cudaMemcpyAsync(h->st.wd + sl * dn, h->host_wd + id * dn, dn, cudaMemcpyHostToDevice, st) == cudaSuccess &&
         cudaMemcpyAsync(h->st.sc + sl * scn, h->host_sc + id * scn, sizeof(float) * scn,
                         cudaMemcpyHostToDevice, st) == cudaSuccess;
    h->slot_owner[sl] = id;
    add(id, sl);
    ++h->copied_records;
    h->copied_bytes += (int64_t)(gu + dn + sizeof(float) * scn);
  }
  flush();
  return ok ? COLI_OK : COLI_ECUDA;
}

// The tier's shape must match the tiered layer: its experts, and n_pin + n_lru HBM slots.
int tier_matches(const coli_moe* h, const coli_tier* tier, int layer, coli_tier_config* tc) {
  if (!h || !tier || !h->hbm_slots) return COLI_EINVAL;
  if (coli_tier_config_of(tier, tc) != COLI_OK || tc->n_experts != h->cfg.n_experts ||
      tc->n_pin + tc->n_lru != h->hbm_slots || layer < 0 || layer >= tc->n_layers)
    return COLI_EINVAL;
  return COLI_OK;
}

// One tiered forward of T <= decode_tmax tokens whose union fits the LRU slots: route and
// publish the selection, read the union back, let the tier manager place its experts, copy the
// misses, then run the expert kernels against the updated slot table.
int run_tiered(coli_moe* h, coli_tier* tier, int layer, const float* x, int T, float* y,
               cudaStream_t st) {
  const Shape s = shape_of(h, T);
  const int E = h->cfg.n_experts;
  cudaError_t e = launch_route(x, s, h->st, h->w, st);
  if (e == cudaSuccess) e = launch_select_publish(s, h->st, h->w, st);
  if (e == cudaSuccess) e = cudaMemcpyAsync(h->pin_union, h->w.n_union, sizeof(int32_t), cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(h->pin_union + 1, h->w.union_ids, sizeof(int32_t) * (E + 1), cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return COLI_ECUDA;
  const int nr = h->pin_union[0] - h->cfg.n_shared;  // routed union experts, ascending ids
  if (nr < 1 || nr > E) return COLI_ECUDA;
  std::vector<int32_t> buf(4 * (size_t)nr);
  int32_t *fi = buf.data(), *fs = fi + nr, *ei = fs + nr, *es = ei + nr;
  int nf = 0, ne = 0;
  int rc = coli_tier_lookup(tier, layer, h->pin_union + 1, nr, nullptr, nullptr, fi, fs, &nf, ei, es, &ne);
  if (rc) return rc;
  if (h->copy_pending) {  // placements made outside a forward land first
    if (cudaStreamWaitEvent(st, h->copy_done, 0) != cudaSuccess) return COLI_ECUDA;
    h->copy_pending = false;
  }
  rc = place(h, ei, es, ne, fi, fs, nf, st);
  if (rc) return rc;
  // the first expert kernel is an ordinary launch: it starts after the slot table update
  ExpertDebug dbg;
  if (T == 1 && h->fused) {
    e = launch_expert_fused(x, y, s, h->st, h->w, dbg, h->num_sms, false, false, st);
  } else {
    e = launch_gateup_decode(s, h->st, h->w, dbg, h->num_sms, false, st);
    if (e == cudaSuccess) e = launch_down_decode(x, y, s, h->st, h->w, dbg, h->num_sms, true, st);
  }
  if (e == cudaSuccess) e = cudaEventRecord(h->fwd_done, st);
  return e == cudaSuccess ? COLI_OK : COLI_ECUDA;
}

// The instantiated host-buffer graph of T tokens, captured on first use on the handle's own
// stream: a kernel that reads x from the mapped pinned staging into the device buffer, the
// forward's launches, and a kernel that writes y and the status word back to the staging (the
// GPU reaches the host memory itself: no copy-engine transfer, whose start-up dominates for a
// few tokens).
int host_graph_for(coli_moe* h, int T, float* dx, float* dy) {
  if (h->host_graph[T]) return COLI_OK;
  if (!h->router_loaded || h->n_loaded < h->slots) return COLI_ESTATE;
  const size_t n = (size_t)T * h->cfg.d;
  cudaStream_t cs = h->cap_stream;
  if (cudaStreamBeginCapture(cs, cudaStreamCaptureModeThreadLocal) != cudaSuccess) return COLI_ECUDA;
  int rc = COLI_OK;
  if (launch_host_in(h->map_x, dx, (int)n, cs) != cudaSuccess) rc = COLI_ECUDA;
  if (rc == COLI_OK) rc = forward_impl(h, dx, T, dy, nullptr, cs);
  if (rc == COLI_OK && launch_host_out(dy, h->map_y, (int)n, h->w.status, h->map_status, cs) != cudaSuccess)
    rc = COLI_ECUDA;
  cudaGraph_t g = nullptr;
  if (cudaStreamEndCapture(cs, &g) != cudaSuccess && rc == COLI_OK) rc = COLI_ECUDA;
  if (rc == COLI_OK && cudaGraphInstantiate(&h->host_graph[T], g, 0) != cudaSuccess) {
    h->host_graph[T] = nullptr;
    rc = COLI_ECUDA;
  }
  if (g) cudaGraphDestroy(g);
  if (rc != COLI_OK) cudaGetLastError();
  return rc;
}

}  // namespace

extern "C" {

int coli_moe_set_prefill_min(coli_moe* h, int min_tokens) {
  if (!h || min_tokens < 2) return COLI_EINVAL;
  h->prefill_min = min_tokens;
  drop_host_graphs(h);  // the cached host-buffer graphs may have taken the other path
  return COLI_OK;
}

int coli_moe_inject_fault(coli_moe* h, int fault) {
  if (!h || (fault != 0 && fault != COLI_FAULT_SKIP_ARRIVAL)) return COLI_EINVAL;
  h->fault = fault;
  return COLI_OK;
}

int coli_moe_launches(const coli_moe* h, int T) {
  if (!h || T < 1 || T > h->cfg.max_tokens) return COLI_EINVAL;
  if (T == 1 && h->fused) return 2;
  if (takes_batched(h, T)) return 8;
  return 3 * ((T + h->decode_tmax - 1) / h->decode_tmax);
}

int64_t coli_moe_expert_record_bytes(int d, int f) {
  return rec_bytes(d, f, 4) + 4LL * (2LL * f + d);
}

int64_t coli_moe_expert_record_bytes_w(int d, int f, int wbits) {
  if (wbits != 4 && wbits != 8 && wbits != 2) return COLI_EINVAL;
  return rec_bytes(d, f, wbits) + 4LL * (2LL * f + d);
}

int coli_moe_create(const coli_moe_config* cfg, coli_moe** out) {
  if (!out) return COLI_EINVAL;
  *out = nullptr;
  if (!cfg) return COLI_EINVAL;
  coli_moe_config c = *cfg;
  if (c.wbits == 0) c.wbits = 4;  // int4 experts unless the caller asks for another width
  if ((c.wbits != 4 && c.wbits != 8 && c.wbits != 2) || c.qblock != 32 || c.n_experts < 1 || c.n_experts > 1024 || c.top_k < 1 ||
      c.top_k > c.n_experts || c.top_k > 32 || (c.n_shared != 0 && c.n_shared != 1) ||
      c.max_tokens < 1 || c.max_tokens > 4096 || !std::isfinite(c.routed_scale) ||
      !(c.rms_eps >= 0.0f) || !std::isfinite(c.rms_eps) || c.d <= 0 || c.f <= 0 ||
      c.hbm_slots < 0)
    return COLI_EINVAL;
  if (c.hbm_slots >= c.n_experts) c.hbm_slots = 0;  // every expert fits: not tiered
  if (c.hbm_slots && c.hbm_slots < c.top_k) return COLI_EINVAL;
  if (!shape_ok(c.d) || !shape_ok(c.f)) return COLI_EUNSUPPORTED;

  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    cudaGetLastError();
    return COLI_ECUDA;
  }
  // tokens per launch of the decode kernels: the largest count up to kDecodeTmax whose
  // shared-memory plans (for the grids they will launch with) leave at least two ring stages
  int decode_tmax = 0;
  for (int Tc = c.max_tokens < kDecodeTmax ? c.max_tokens : kDecodeTmax; Tc >= 1 && !decode_tmax; --Tc) {
    const long slots = (long)(Tc * c.top_k < c.n_experts ? Tc * c.top_k : c.n_experts) + c.n_shared;
    const long gu_grid = slots * (c.f / 32) < sms ? slots * (c.f / 32) : sms;
    const int dn_grid = down_grid(c.d, sms);
    if (gateup_plan(c.d, c.f, Tc, c.top_k, c.n_experts, c.n_shared, (int)gu_grid, c.wbits).nst >= 2 &&
        down_plan(c.d, c.f, Tc, c.top_k, c.n_experts, c.n_shared, (int)dn_grid, c.wbits).nst >= 2)
      decode_tmax = Tc;
  }
  if (!decode_tmax) return COLI_EUNSUPPORTED;
  if (configure_device(dev) != cudaSuccess) {
    cudaGetLastError();
    return COLI_ECUDA;
  }

  coli_moe* h = new (std::nothrow) coli_moe();
  if (!h) return COLI_ENOMEM;
  h->cfg = c;
  h->device = dev;
  if (cudaDeviceGetAttribute(&h->num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    delete h;
    return COLI_ECUDA;
  }
  h->slots = c.n_experts + c.n_shared;
  h->decode_tmax = decode_tmax;
  h->hbm_slots = c.hbm_slots;
  h->loaded.assign(h->slots, 0);
  // the fused one-token kernel and the tensor-core path take int4 experts
  h->fused = c.wbits == 4 && fused_supported(c.d, c.f, c.top_k, c.n_experts, c.n_shared, h->num_sms);
  // device store slots: every expert, or a tiered layer's routed slots and the shared one
  const long S = h->hbm_slots ? h->hbm_slots + c.n_shared : h->slots;
  const long d = c.d, f = c.f, E = c.n_experts, K = c.top_k, Tm = c.max_tokens;
  const long Pm = Tm * K + (c.n_shared ? Tm : 0);
  int rc = COLI_OK;
#define ALLOC(ptr, bytes) \
  if (rc == COLI_OK) rc = dalloc(h, &(ptr), (size_t)(bytes));
  const long wb = c.wbits;
  ALLOC(h->st.wgu, S * f * (2 * d * wb / 8))
  ALLOC(h->st.wd, S * d * (f * wb / 8))
  ALLOC(h->st.sc, sizeof(float) * S * (2 * f + d))
  ALLOC(h->st.wr, sizeof(float) * E * d)
  if (c.has_norm) ALLOC(h->st.gamma, sizeof(float) * d)
  ALLOC(h->w.xn, sizeof(float) * Tm * d)
  ALLOC(h->w.xnp, sizeof(float) * Tm * d)
  ALLOC(h->w.qx, Tm * d)
  ALLOC(h->w.dx, sizeof(float) * Tm * (d / 32))
  ALLOC(h->w.sx, sizeof(int32_t) * Tm * (d / 32))
  ALLOC(h->w.logits, sizeof(float) * Tm * E)
  ALLOC(h->w.scores, sizeof(float) * Tm * E)
  ALLOC(h->w.ids, sizeof(int32_t) * Tm * K)
  ALLOC(h->w.w, sizeof(float) * Tm * K)
  ALLOC(h->w.n_union, sizeof(int32_t) * 4)
  ALLOC(h->w.union_ids, sizeof(int32_t) * (E + 1))
  ALLOC(h->w.offsets, sizeof(int32_t) * (E + 2))
  ALLOC(h->w.pair_token, sizeof(int32_t) * Pm)
  ALLOC(h->w.pair_rank, sizeof(int32_t) * Pm)
  ALLOC(h->w.inv, sizeof(int32_t) * Tm * K)
  ALLOC(h->w.hf, sizeof(float) * (Pm + kPrefillTileN) * f)
  ALLOC(h->w.qh, (Pm + kPrefillTileN) * f)
  ALLOC(h->w.dh, sizeof(float) * (Pm + kPrefillTileN) * (f / 32))
  ALLOC(h->w.sh, sizeof(int32_t) * Pm * (f / 32))
  ALLOC(h->w.sel_flag, sizeof(int32_t) * 4)
  ALLOC(h->w.status, sizeof(int32_t) * 4)
  ALLOC(h->dev_io, sizeof(float) * 2 * Tm * d)
  if (h->hbm_slots) {
    // tiered: the slot table (nothing routed resident yet, the shared expert in the slot after
    // the routed ones), every record's pinned host copy, the union read-back buffer, events
    ALLOC(h->slot_of, sizeof(int32_t) * (E + 1))
    std::vector<int32_t> init((size_t)E + 1, -1);
    if (c.n_shared) init[E] = h->hbm_slots;
    if (rc == COLI_OK && cudaMemcpy(h->slot_of, init.data(), sizeof(int32_t) * (E + 1),
                                    cudaMemcpyHostToDevice) != cudaSuccess)
      rc = COLI_ECUDA;
    h->st.slot_of = h->slot_of;
    h->slot_owner.assign((size_t)S, -1);
    if (c.n_shared) h->slot_owner[h->hbm_slots] = (int32_t)E;
    const size_t n1 = (size_t)h->slots;
    const size_t sizes[4] = {n1 * f * (2 * d * wb / 8), n1 * d * (f * wb / 8), sizeof(float) * n1 * (2 * f + d),
                             sizeof(int32_t) * (E + 2)};
    void* ptrs[4] = {};
    for (int i = 0; i < 4 && rc == COLI_OK; ++i) {
      if (cudaHostAlloc(&ptrs[i], sizes[i], cudaHostAllocDefault) != cudaSuccess) {
        cudaGetLastError();
        rc = COLI_ENOMEM;
      } else {
        h->host_allocs.push_back(ptrs[i]);
      }
    }
    h->host_wgu = static_cast<uint8_t*>(ptrs[0]);
    h->host_wd = static_cast<uint8_t*>(ptrs[1]);
    h->host_sc = static_cast<float*>(ptrs[2]);
    h->pin_union = static_cast<int32_t*>(ptrs[3]);
    if (rc == COLI_OK && (cudaEventCreateWithFlags(&h->copy_done, cudaEventDisableTiming) != cudaSuccess ||
                          cudaEventCreateWithFlags(&h->fwd_done, cudaEventDisableTiming) != cudaSuccess))
      rc = COLI_ECUDA;
  }
  // the tensor-core path takes int4 layers whose every expert is resident
  if (rc == COLI_OK && c.wbits == 4 && !h->hbm_slots && Tm > kDecodeTmax && d % 256 == 0 &&
      configure_prefill_kernels((int)d, (int)f, (int)E) == cudaSuccess &&
      configure_route_batch_kernels((int)E) == cudaSuccess) {
    const long prow = Pm + kPrefillTileN;
    ALLOC(h->pw.xb, sizeof(__nv_bfloat16) * prow * d)
    ALLOC(h->pw.dxp, sizeof(float) * prow * (d / 32))
    ALLOC(h->pw.hb, sizeof(__nv_bfloat16) * prow * f)
    ALLOC(h->pw.e, sizeof(float) * Pm * d)
    ALLOC(h->pw.tile_prefix, sizeof(int32_t) * (E + 2))
    if (rc == COLI_OK) {
      h->prefill = prefill_make_maps(&h->maps, h->st, h->w, h->pw, (int)d, (int)f, (int)E, (int)S,
                                     (int)prow, (int)Tm);
      if (cudaMemset(h->pw.xb, 0, sizeof(__nv_bfloat16) * prow * d) != cudaSuccess ||
          cudaMemset(h->pw.hb, 0, sizeof(__nv_bfloat16) * prow * f) != cudaSuccess ||
          cudaMemset(h->pw.dxp, 0, sizeof(float) * prow * (d / 32)) != cudaSuccess)
        rc = COLI_ECUDA;
    }
  }
#undef ALLOC
  if (rc == COLI_OK) {
    const size_t n = (size_t)(Tm < kHostGraphMaxT ? Tm : kHostGraphMaxT) * d;
    void* p = nullptr;
    void* q = nullptr;
    if (cudaHostAlloc(&p, sizeof(float) * 2 * n + 64, cudaHostAllocMapped) != cudaSuccess) {
      cudaGetLastError();
      rc = COLI_ENOMEM;
    } else {
      h->pin_x = static_cast<float*>(p);
      h->pin_y = h->pin_x + n;
      h->pin_status = reinterpret_cast<int32_t*>(h->pin_y + n);
      *h->pin_status = 0;
      h->pin_status[kHostDoneWord] = 0;
      h->host_done = 0;
      if (cudaHostGetDevicePointer(&q, p, 0) != cudaSuccess ||
          cudaStreamCreateWithFlags(&h->cap_stream, cudaStreamNonBlocking) != cudaSuccess) {
        cudaGetLastError();
        rc = COLI_ECUDA;
      } else {
        h->map_x = static_cast<float*>(q);
        h->map_y = h->map_x + n;
        h->map_status = reinterpret_cast<int32_t*>(h->map_y + n);
      }
    }
  }
  if (rc == COLI_OK && (cudaMemset(h->w.sel_flag, 0, 16) != cudaSuccess ||
                        cudaMemset(h->w.status, 0, 16) != cudaSuccess ||
                        cudaDeviceSynchronize() != cudaSuccess))
    rc = COLI_ECUDA;
  if (rc != COLI_OK) {
    free_all(h);
    delete h;
    return rc;
  }
  *out = h;
  return COLI_OK;
}

void coli_moe_destroy(coli_moe* h) {
  if (!h) return;
  cudaDeviceSynchronize();
  free_all(h);
  delete h;
}

int coli_moe_load_router(coli_moe* h, const float* W_r, const float* bias, const float* gamma,
                         void* stream) {
  if (!h || !W_r) return COLI_EINVAL;
  if (h->cfg.has_norm && !gamma) return COLI_EINVAL;
  int rc = check_device(h);
  if (rc) return rc;
  cudaStream_t st = (cudaStream_t)stream;
  const size_t E = h->cfg.n_experts, d = h->cfg.d;
  float* tmp = nullptr;
  if (cudaMalloc(&tmp, sizeof(float) * E * d) != cudaSuccess) {
    cudaGetLastError();
    return COLI_ENOMEM;
  }
  cudaError_t e = cudaMemcpyAsync(tmp, W_r, sizeof(float) * E * d, cudaMemcpyDefault, st);
  if (e == cudaSuccess) e = launch_permute_router(tmp, h->st.wr, (int)E, (int)d, st);
  if (e == cudaSuccess && bias) {
    if (!h->st.bias) {
      if (dalloc(h, &h->st.bias, sizeof(float) * E) != COLI_OK) {
        cudaStreamSynchronize(st);
        cudaFree(tmp);
        return COLI_ENOMEM;
      }
    }
    e = cudaMemcpyAsync(h->st.bias, bias, sizeof(float) * E, cudaMemcpyDefault, st);
  }
  if (e == cudaSuccess && h->cfg.has_norm)
    e = cudaMemcpyAsync(h->st.gamma, gamma, sizeof(float) * d, cudaMemcpyDefault, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  cudaFree(tmp);
  if (e != cudaSuccess) return COLI_ECUDA;
  if (!bias && h->st.bias) {
    // a later load without bias removes it
    for (size_t i = 0; i < h->allocs.size(); ++i)
      if (h->allocs[i] == h->st.bias) {
        cudaFree(h->st.bias);
        h->allocs.erase(h->allocs.begin() + i);
        break;
      }
    h->st.bias = nullptr;
  }
  h->router_loaded = true;
  drop_host_graphs(h);  // the cached host-buffer graphs hold the old bias pointer
  return COLI_OK;
}

int coli_moe_load_experts(coli_moe* h, int first, int count, const uint8_t* packed,
                          const float* scales, void* stream) {
  if (!h || !packed || !scales || first < 0 || count < 0 || first + count > h->slots)
    return COLI_EINVAL;
  if (count == 0) return COLI_OK;
  int rc = check_device(h);
  if (rc) return rc;
  cudaStream_t st = (cudaStream_t)stream;
  const int d = h->cfg.d, f = h->cfg.f, wb = h->cfg.wbits;
  const size_t rb = (size_t)rec_bytes(d, f, wb);
  const size_t rbd = (size_t)d * wb / 8, rbf = (size_t)f * wb / 8;  // bytes of a gate/up, a down row
  const size_t mat = (size_t)f * rbd;                                 // bytes of a gate or up matrix
  const bool on_device = is_device_ptr(packed);
  const bool tiered = h->hbm_slots > 0;
  const size_t scn = (size_t)(2 * f + d);  // scales of a record
  uint8_t* staging = nullptr;  // a host record on the device
  uint8_t* rstage = nullptr;   // tiered: one record in the store layout, on its way to the host
  if (!on_device && cudaMalloc(&staging, rb) != cudaSuccess) {
    cudaGetLastError();
    return COLI_ENOMEM;
  }
  if (tiered && cudaMalloc(&rstage, 2 * mat + (size_t)d * rbf) != cudaSuccess) {
    cudaGetLastError();
    if (staging) cudaFree(staging);
    return COLI_ENOMEM;
  }
  cudaError_t e = cudaSuccess;
  for (int i = 0; i < count && e == cudaSuccess; ++i) {
    const int id = first + i;
    const uint8_t* rec = packed + (size_t)i * rb;
    if (!on_device) {
      e = cudaMemcpyAsync(staging, rec, rb, cudaMemcpyHostToDevice, st);
      if (e == cudaSuccess) e = cudaStreamSynchronize(st);
      rec = staging;
    }
    // gate row r and up row r side by side (row pairs), then the down rows: into the expert's
    // device slot, or (tiered) into the staging record that then goes to the pinned host copy
    uint8_t* gu = tiered ? rstage : h->st.wgu + (size_t)id * 2 * mat;
    uint8_t* dn = tiered ? rstage + 2 * mat : h->st.wd + (size_t)id * d * rbf;
    if (e == cudaSuccess) e = launch_repack_matrix(rec, gu, f, d, 2 * rbd, st, wb);
    if (e == cudaSuccess) e = launch_repack_matrix(rec + mat, gu + rbd, f, d, 2 * rbd, st, wb);
    if (e == cudaSuccess) e = launch_repack_matrix(rec + 2 * mat, dn, d, f, rbf, st, wb);
    if (!tiered) {
      if (e == cudaSuccess)
        e = cudaMemcpyAsync(h->st.sc + (size_t)id * scn, scales + (size_t)i * scn, sizeof(float) * scn,
                            cudaMemcpyDefault, st);
      continue;
    }
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(h->host_wgu + (size_t)id * 2 * mat, rstage, 2 * mat, cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(h->host_wd + (size_t)id * d * rbf, rstage + 2 * mat, (size_t)d * rbf,
                          cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(h->host_sc + (size_t)id * scn, scales + (size_t)i * scn, sizeof(float) * scn,
                          cudaMemcpyDefault, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);  // the staging record is reused
    // a record that is resident (the shared expert always is) gets the new bytes in HBM too
    for (size_t sl = 0; sl < h->slot_owner.size() && e == cudaSuccess; ++sl) {
      if (h->slot_owner[sl] != id) continue;
      e = cudaMemcpyAsync(h->st.wgu + sl * 2 * mat, h->host_wgu + (size_t)id * 2 * mat, 2 * mat,
                          cudaMemcpyHostToDevice, st);
      if (e == cudaSuccess)
        e = cudaMemcpyAsync(h->st.wd + sl * d * rbf, h->host_wd + (size_t)id * d * rbf, (size_t)d * rbf,
                            cudaMemcpyHostToDevice, st);
      if (e == cudaSuccess)
        e = cudaMemcpyAsync(h->st.sc + sl * scn, h->host_sc + (size_t)id * scn, sizeof(float) * scn,
                            cudaMemcpyHostToDevice, st);
    }
  }
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (staging) cudaFree(staging);
  if (rstage) cudaFree(rstage);
  if (e != cudaSuccess) return COLI_ECUDA;
  for (int i = 0; i < count; ++i)
    if (!h->loaded[first + i]) {
      h->loaded[first + i] = 1;
      ++h->n_loaded;
    }
  return COLI_OK;
}

int coli_moe_forward(coli_moe* h, const float* x_dev, int T, float* y_dev, void* stream) {
  return forward_impl(h, x_dev, T, y_dev, nullptr, stream);
}

int coli_moe_forward_debug(coli_moe* h, const float* x_dev, int T, float* y_dev,
                           const coli_moe_dump* dump, void* stream) {
  if (!dump) return COLI_EINVAL;
  return forward_impl(h, x_dev, T, y_dev, dump, stream);
}

int coli_moe_forward_profiled(coli_moe* h, const float* x_dev, int T, float* y_dev,
                              void* const* events, int n_events, void* stream) {
  if (!h || !events || n_events < 4 || T < 1 || T > h->cfg.max_tokens) return COLI_EINVAL;
  const bool batched = takes_batched(h, T);
  if (T > h->decode_tmax && !batched) return COLI_EINVAL;
  for (int i = 0; i < 4; ++i)
    if (!events[i]) return COLI_EINVAL;
  if (!x_dev || !y_dev || ((uintptr_t)x_dev & 15u) || ((uintptr_t)y_dev & 3u)) return COLI_EINVAL;
  const size_t bytes = sizeof(float) * (size_t)T * h->cfg.d;
  if (x_dev != y_dev && overlap(x_dev, bytes, y_dev, bytes)) return COLI_EINVAL;
  if (x_dev == y_dev && !h->cfg.has_norm) return COLI_EINVAL;
  if (!h->router_loaded || h->n_loaded < h->slots) return COLI_ESTATE;
  int rc = check_device(h);
  if (rc) return rc;
  cudaEvent_t ev[4];
  for (int i = 0; i < 4; ++i) ev[i] = (cudaEvent_t)events[i];
  if (batched) return run_prefill(h, x_dev, T, y_dev, nullptr, (cudaStream_t)stream, ev);
  return run_decode(h, x_dev, T, y_dev, nullptr, (cudaStream_t)stream, ev);
}

int coli_moe_forward_host(coli_moe* h, const float* x_host, int T, float* y_host, void* stream) {
  if (!h || T < 0 || T > h->cfg.max_tokens) return COLI_EINVAL;
  if (T == 0) return COLI_OK;
  if (!x_host || !y_host) return COLI_EINVAL;
  int rc = check_device(h);
  if (rc) return rc;
  cudaStream_t st = (cudaStream_t)stream;
  const size_t n = (size_t)T * h->cfg.d;
  float* dx = h->dev_io;
  float* dy = h->cfg.has_norm ? h->dev_io : h->dev_io + (size_t)h->cfg.max_tokens * h->cfg.d;
  if (T <= kHostGraphMaxT && !h->fault && !h->hbm_slots) {
    // small batch: x into the pinned staging, one graph launch (copy in, kernels, copy out,
    // status word), one synchronisation, y out of the staging
    rc = host_graph_for(h, T, dx, dy);
    if (rc) return rc;
    memcpy(h->pin_x, x_host, sizeof(float) * n);
    if (cudaGraphLaunch(h->host_graph[T], st) != cudaSuccess) return COLI_ECUDA;
    // the graph's last kernel writes y and the status word, then raises the completion counter:
    // poll it (an acquire load, so y is read after it) instead of a stream synchronisation; past
    // a second, or on any mismatch, fall back to the synchronisation and resume from the counter
    const int32_t want = h->host_done + 1;
    const auto t0 = std::chrono::steady_clock::now();
    bool seen = false;
    for (uint32_t it = 1;; ++it) {
      if (__atomic_load_n(h->pin_status + kHostDoneWord, __ATOMIC_ACQUIRE) == want) {
        seen = true;
        break;
      }
      if ((it & 1023u) == 0 && std::chrono::steady_clock::now() - t0 > std::chrono::seconds(1)) break;
    }
    if (!seen) {
      if (cudaStreamSynchronize(st) != cudaSuccess) return COLI_ECUDA;
      h->host_done = __atomic_load_n(h->pin_status + kHostDoneWord, __ATOMIC_ACQUIRE);
    } else {
      h->host_done = want;
    }
    memcpy(y_host, h->pin_y, sizeof(float) * n);
    // a bounded device wait that gave up leaves y undefined: report it (and clear it) here
    return *h->pin_status == COLI_OK ? COLI_OK : coli_moe_status(h, stream);
  }
  if (cudaMemcpyAsync(dx, x_host, sizeof(float) * n, cudaMemcpyHostToDevice, st) != cudaSuccess)
    return COLI_ECUDA;
  rc = forward_impl(h, dx, T, dy, nullptr, stream);
  if (rc) return rc;
  if (cudaMemcpyAsync(y_host, dy, sizeof(float) * n, cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return COLI_ECUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return COLI_ECUDA;
  // the call has synchronised anyway: report a bounded device wait that gave up (y_host is then
  // undefined) instead of leaving it for coli_moe_status
  return coli_moe_status(h, stream);
}

int coli_moe_forward_tiered(coli_moe* h, coli_tier* tier, int layer, const float* x_dev, int T,
                            float* y_dev, void* stream) {
  coli_tier_config tc;
  int rc = tier_matches(h, tier, layer, &tc);
  if (rc) return rc;
  if (T < 0 || T > h->cfg.max_tokens) return COLI_EINVAL;
  if (T == 0) return COLI_OK;
  if (!x_dev || !y_dev || ((uintptr_t)x_dev & 15u) || ((uintptr_t)y_dev & 3u)) return COLI_EINVAL;
  const size_t bytes = sizeof(float) * (size_t)T * h->cfg.d;
  if (x_dev != y_dev && overlap(x_dev, bytes, y_dev, bytes)) return COLI_EINVAL;
  if (x_dev == y_dev && !h->cfg.has_norm) return COLI_EINVAL;
  if (!h->router_loaded || h->n_loaded < h->slots) return COLI_ESTATE;
  if ((rc = check_device(h))) return rc;
  // a chunk's routed union must fit the LRU slots: at most n_lru / K tokens at a time
  int tm = tc.n_lru / h->cfg.top_k;
  if (tm > h->decode_tmax) tm = h->decode_tmax;
  if (tm < 1) return COLI_EUNSUPPORTED;
  cudaStream_t st = (cudaStream_t)stream;
  for (int c0 = 0; c0 < T; c0 += tm) {
    const int Tc = T - c0 < tm ? T - c0 : tm;
    rc = run_tiered(h, tier, layer, x_dev + (size_t)c0 * h->cfg.d, Tc, y_dev + (size_t)c0 * h->cfg.d, st);
    if (rc) return rc;
  }
  return COLI_OK;
}

int coli_moe_prefetch_tiered(coli_moe* h, coli_tier* tier, int layer, const int32_t* ids, int n,
                             void* stream) {
  coli_tier_config tc;
  int rc = tier_matches(h, tier, layer, &tc);
  if (rc) return rc;
  if (n < 0 || (n > 0 && !ids)) return COLI_EINVAL;
  if (n == 0) return COLI_OK;
  if ((rc = check_device(h))) return rc;
  std::vector<int32_t> buf(4 * (size_t)n);
  int32_t *fi = buf.data(), *fs = fi + n, *ei = fs + n, *es = ei + n;
  int nf = 0, ne = 0;
  if ((rc = coli_tier_prefetch(tier, layer, ids, n, fi, fs, &nf, ei, es, &ne))) return rc;
  if (nf + ne == 0) return COLI_OK;
  cudaStream_t st = (cudaStream_t)stream;
  // no copy may overwrite a slot that an earlier forward still reads
  if (cudaStreamWaitEvent(st, h->fwd_done, 0) != cudaSuccess) return COLI_ECUDA;
  if ((rc = place(h, ei, es, ne, fi, fs, nf, st))) return rc;
  if (cudaEventRecord(h->copy_done, st) != cudaSuccess) return COLI_ECUDA;
  h->copy_pending = true;
  return COLI_OK;
}

int coli_moe_repin_tiered(coli_moe* h, coli_tier* tier, int layer, int by_usage, void* stream) {
  coli_tier_config tc;
  int rc = tier_matches(h, tier, layer, &tc);
  if (rc) return rc;
  if ((rc = check_device(h))) return rc;
  const int m = tc.n_pin > 0 ? tc.n_pin : 1;
  std::vector<int32_t> buf(4 * (size_t)m);
  int32_t *fi = buf.data(), *fs = fi + m, *di = fs + m, *ds = di + m;
  int nf = 0, nd = 0;
  rc = by_usage ? coli_tier_autopin(tier, layer, fi, fs, &nf, di, ds, &nd)
                : coli_tier_repin(tier, layer, fi, fs, &nf, di, ds, &nd);
  if (rc) return rc;
  if (nf + nd == 0) return COLI_OK;
  cudaStream_t st = (cudaStream_t)stream;
  if (cudaStreamWaitEvent(st, h->fwd_done, 0) != cudaSuccess) return COLI_ECUDA;
  if ((rc = place(h, di, ds, nd, fi, fs, nf, st))) return rc;
  if (cudaEventRecord(h->copy_done, st) != cudaSuccess) return COLI_ECUDA;
  h->copy_pending = true;
  return COLI_OK;
}

int coli_moe_tier_copies(const coli_moe* h, int64_t* records, int64_t* bytes) {
  if (!h || !records || !bytes) return COLI_EINVAL;
  *records = h->copied_records;
  *bytes = h->copied_bytes;
  return COLI_OK;
}

int coli_moe_stack_forward(coli_moe* const* layers, int n_layers, float* x_dev, int T,
                           void* stream) {
  if (!layers || n_layers < 0 || !x_dev) return COLI_EINVAL;
  for (int l = 0; l < n_layers; ++l) {
    if (!layers[l] || !layers[l]->cfg.has_norm || layers[l]->cfg.d != layers[0]->cfg.d)
      return COLI_EINVAL;
  }
  for (int l = 0; l < n_layers; ++l) {
    const int rc = forward_impl(layers[l], x_dev, T, x_dev, nullptr, stream);
    if (rc) return rc;
  }
  return COLI_OK;
}

int coli_moe_status(coli_moe* h, void* stream) {
  if (!h) return COLI_EINVAL;
  int rc = check_device(h);
  if (rc) return rc;
  cudaStream_t st = (cudaStream_t)stream;
  int32_t v = 0;
  if (cudaMemcpyAsync(&v, h->w.status, sizeof(v), cudaMemcpyDeviceToHost, st) != cudaSuccess ||
      cudaStreamSynchronize(st) != cudaSuccess)
    return COLI_ECUDA;
  if (v != COLI_OK) {
    // clear the status and the selection flag together
    if (cudaMemset(h->w.status, 0, 16) != cudaSuccess || cudaMemset(h->w.sel_flag, 0, 16) != cudaSuccess ||
        cudaDeviceSynchronize() != cudaSuccess)
      return COLI_ECUDA;
    return v;
  }
  return COLI_OK;
}

int coli_quantize_i4_rows(const float* w_dev, int64_t rows, int cols, uint8_t* packed_dev,
                          float* scales_dev, void* stream) {
  if (rows < 0 || cols <= 0 || cols % 2 || cols > 65536) return COLI_EINVAL;
  if (rows == 0) return COLI_OK;
  if (!w_dev || !packed_dev || !scales_dev) return COLI_EINVAL;
  return cuda_status(
      launch_quantize_i4_rows(w_dev, rows, cols, packed_dev, scales_dev, (cudaStream_t)stream));
}

int coli_quantize_i8_rows(const float* w_dev, int64_t rows, int cols, int8_t* q_dev,
                          float* scales_dev, void* stream) {
  if (rows < 0 || cols <= 0 || cols > 65536) return COLI_EINVAL;
  if (rows == 0) return COLI_OK;
  if (!w_dev || !q_dev || !scales_dev) return COLI_EINVAL;
  return cuda_status(
      launch_quantize_i8_rows(w_dev, rows, cols, q_dev, scales_dev, (cudaStream_t)stream));
}

int coli_quantize_i2_rows(const float* w_dev, int64_t rows, int cols, uint8_t* packed_dev,
                          float* scales_dev, void* stream) {
  if (rows < 0 || cols <= 0 || cols % 4 || cols > 65536) return COLI_EINVAL;
  if (rows == 0) return COLI_OK;
  if (!w_dev || !packed_dev || !scales_dev || ((uintptr_t)w_dev & 15u)) return COLI_EINVAL;
  return cuda_status(
      launch_quantize_i2_rows(w_dev, rows, cols, packed_dev, scales_dev, (cudaStream_t)stream));
}

int coli_quantize_act_q8(const float* x_dev, int64_t n, int8_t* q_dev, float* d_dev,
                         void* stream) {
  if (n < 0 || n % 32) return COLI_EINVAL;
  if (n == 0) return COLI_OK;
  if (!x_dev || !q_dev || !d_dev) return COLI_EINVAL;
  return cuda_status(launch_quantize_q8(x_dev, n, q_dev, d_dev, (cudaStream_t)stream));
}

}  // extern "C"
