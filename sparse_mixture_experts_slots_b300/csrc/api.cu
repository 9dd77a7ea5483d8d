// C ABI of the Switch MoE layer: argument checks, workspace, stage launches.
// The operations are specified in include/switch_moe.h.
#include <math.h>
#include <stdlib.h>
#include <string.h>

#include <algorithm>
#include <new>

#include "../../include/switch_moe.h"
#include "common.cuh"
#include "kernels.h"

using namespace smoe;

// Resources of switch_forward_host, created by its first call: a copy-in and a copy-out
// stream, two staging slots (x, y, aux loss) that alternate between calls, and the events
// that keep a slot from being reused while a copy or the layer still reads it.
struct HostPath {
  cudaStream_t cin, cout;
  cudaEvent_t in_done[2], fwd_done[2], out_done[2];
  uint8_t* stage;     // x[2], y[2] (act_bytes each, 256-aligned), aux[2] (256 B each)
  size_t act_bytes, slot_stride;
  unsigned calls;
  int n_events;       // events created (for cleanup)
  bool ok;
};

struct switch_layer {
  switch_config cfg;
  int N, C, Ceff, R, nT;
  int es;  // bytes per act element
  int device;
  uint8_t* ws;
  size_t ws_bytes;
  uint32_t* err;
  float* logits;
  int32_t* tile_hist;
  float* tile_P;
  float* tile_Z;
  int32_t* tile_base;
  int32_t* tile_hist2;  // top-2 only
  int32_t* tile_base2;
  int32_t* group_off;
  int32_t* tok_of_row;
  void* wsplit;
  void* xchg;  // the router's global exchange rows, or null
  uint32_t* ffn_counters;
  int ffn_counter_words;
  float* scan_partial;
  uint32_t* scan_counter;
  void* xe;
  void* hbuf;
  void* ye;
  // backward scratch (SWITCH_FLAG_TRAINING): float32
  float* bw_dye;  // [E, R, d]
  float* bw_dh;   // [E, R, F]
  float* bw_dxe;  // [E, R, d]
  float* bw_dg;   // [N]
  float* bw_dz;   // [N, E]
  float* bw_part; // [nsplit, E, d]: per-token-chunk partial sums of dWr and dbr (or [ntc, 2E, d])
  int bw_nsplit;
  int bw_ntc, bw_kc;          // tensor-core router products: token chunks and their rows (ntc 0: off)
  void* bw_dzp;               // [N, 3E] bf16
  void* bw_Wp;                // [3E, d] bf16
  int32_t* bw_rows_k;         // [ntc + 1]
  // tensor-core backward (bf16 with tensor-core FFN shapes): bf16 copies of the gradients
  bool bw_tc;
  void* bw_dye16; // [E, R, d]
  void* bw_dh16;  // [E, R, F]
  void* bw_dxe16; // [E, R, d]
  int bw_Rpad;
  int32_t* bw_rows_d; int32_t* bw_rows_F;
  uint32_t* bw_counters; int bw_counter_words;
  bool wsplit_ready;  // wsplit holds the pieces of the last router weights split on this handle
  int route_ctas, ffn_ctas;  // CTA caps of the persistent router and FFN kernels (0: none)
  cudaEvent_t ev[6];
  bool have_events;
  int last_launches;
  HostPath* hp;
};

namespace {

constexpr int MAX_E = 2048;

bool top2_of(const switch_config* c) { return (c->flags & SWITCH_FLAG_TOP2) != 0; }
bool training_of(const switch_config* c) { return (c->flags & SWITCH_FLAG_TRAINING) != 0; }

int64_t capacity_of(const switch_config* c) {
  if (c->capacity_override > 0) return c->capacity_override;
  if (c->T <= 0) return 0;
  // top-2: twice top-1's capacity (each token makes two requests)
  const double v = (top2_of(c) ? 2.0 : 1.0) * c->capacity_factor * (double)c->T / (double)c->E;
  const double r = nearbyint(v);
  if (fabs(v - r) <= 1e-9) return (int64_t)r;
  return (int64_t)ceil(v);
}

bool config_ok(const switch_config* c) {
  if (!c) return false;
  if (c->G < 1 || c->T < 0 || c->d_model < 1 || c->d_ff < 1 || c->E < 1 || c->E > MAX_E) return false;
  if (top2_of(c) && c->E < 2) return false;
  if (c->dtype != SWITCH_F32 && c->dtype != SWITCH_BF16) return false;
  if (c->capacity_override < 0) return false;
  if (c->capacity_override == 0 && !(c->capacity_factor > 0.0 && c->capacity_factor < 1e6)) return false;
  const int es = c->dtype == SWITCH_F32 ? 4 : 2;
  if ((c->d_model * es) % 16 != 0 || (c->d_ff * es) % 16 != 0) return false;
  const int64_t N = (int64_t)c->G * c->T;
  if (N > (int64_t)1 << 30) return false;
  if (N * c->E > (int64_t)1 << 36) return false;
  const int64_t C = capacity_of(c);
  const int64_t Ceff = C < c->T ? C : c->T;
  if ((int64_t)c->G * Ceff * c->E > (int64_t)1 << 30) return false;
  // grid limits: routing groups on grid.y, token tiles of 64 rows of one expert block on grid.y
  if (c->G > 65535 || (int64_t)c->G * Ceff > (int64_t)65535 * 64 || N > (int64_t)65535 * 64) return false;
  return true;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Per-token arrays may be NULL only when there are no tokens.
bool route_out_ok(const switch_route_out* r, int64_t N, bool top2 = false) {
  if (!r) return false;
  if (N > 0 && !(r->expert && r->slot && r->keep && r->gate && r->row)) return false;
  if (top2 && N > 0 && !(r->expert2 && r->slot2 && r->keep2 && r->gate2 && r->row2)) return false;
  if (top2 && !(r->raw2_count && r->accepted2_count)) return false;
  return r->raw_count && r->accepted_count && r->P && r->balance && r->aux_loss_per_group && r->aux_loss &&
         r->expert_rows;
}

switch_status launched(int n, switch_layer* h) {
  if (n < 0) return SWITCH_ERR_CUDA;
  h->last_launches += n;
  return SWITCH_OK;
}

}  // namespace

extern "C" {

int64_t switch_capacity(const switch_config* cfg) { return config_ok(cfg) ? capacity_of(cfg) : -1; }

int64_t switch_expert_block_rows(const switch_config* cfg) {
  if (!config_ok(cfg)) return -1;
  const int64_t C = capacity_of(cfg);
  return (int64_t)cfg->G * (C < cfg->T ? C : cfg->T);
}

const char* switch_status_string(switch_status s) {
  switch (s) {
    case SWITCH_OK: return "ok";
    case SWITCH_ERR_INVALID_ARG: return "invalid argument";
    case SWITCH_ERR_UNSUPPORTED: return "unsupported";
    case SWITCH_ERR_CUDA: return "CUDA error";
    case SWITCH_ERR_DEVICE_TIMEOUT: return "device wait timed out";
    case SWITCH_ERR_OOM: return "out of device memory";
    case SWITCH_ERR_DEVICE_BOUNDS: return "device bounds check failed";
  }
  return "unknown status";
}

switch_status switch_create(const switch_config* cfg, switch_handle* out) {
  if (!out) return SWITCH_ERR_INVALID_ARG;
  *out = nullptr;
  if (!config_ok(cfg)) return SWITCH_ERR_INVALID_ARG;
  switch_layer* h = new (std::nothrow) switch_layer();
  if (!h) return SWITCH_ERR_OOM;
  h->cfg = *cfg;
  h->N = cfg->G * cfg->T;
  h->C = (int)capacity_of(cfg);
  h->Ceff = h->C < cfg->T ? h->C : cfg->T;
  h->R = cfg->G * h->Ceff;
  h->nT = (cfg->T + ROUTE_TILE - 1) / ROUTE_TILE;
  h->es = cfg->dtype == SWITCH_F32 ? 4 : 2;
  if (cudaGetDevice(&h->device) != cudaSuccess) {
    delete h;
    return SWITCH_ERR_CUDA;
  }
  const size_t E = cfg->E, G = cfg->G, N = h->N, R = h->R, nT = h->nT;
  const size_t d = cfg->d_model, F = cfg->d_ff;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = round_up(off + bytes, 256);
    return o;
  };
  const size_t o_err = take(sizeof(uint32_t) * 4);  // [0] error word, [1] scan counter
  // float32 logits are materialised only by the CUDA-core router (float32 activations)
  const bool two = top2_of(cfg);
  const bool train = training_of(cfg);
  const size_t o_logits = take(cfg->dtype == SWITCH_F32 || two || train ? N * E * sizeof(float) : 0);
  const size_t o_wsplit = take(cfg->dtype == SWITCH_BF16 ? router_tc_wsplit_bytes(cfg->E, cfg->d_model) : 0);
  const size_t xchg_bytes =
      cfg->dtype == SWITCH_BF16 ? router_tc_exchange_bytes((long long)(G * nT), cfg->E, two) : 0;
  const size_t o_xchg = take(xchg_bytes);
  const size_t o_part = take(G * (size_t)route_scan_blocks(cfg->E) * sizeof(float));
  const size_t ffn_words = ffn_counter_words(cfg->E, (int)R, cfg->d_model, cfg->d_ff);
  const size_t o_fcnt = take(ffn_words * sizeof(uint32_t));
  const size_t o_hist = take(G * nT * E * sizeof(int32_t));
  const size_t o_tP = take(G * nT * E * sizeof(float));
  const size_t o_tZ = take(G * nT * sizeof(float));
  const size_t o_base = take(G * nT * E * sizeof(int32_t));
  const size_t o_hist2 = take(two ? G * nT * E * sizeof(int32_t) : 0);
  const size_t o_base2 = take(two ? G * nT * E * sizeof(int32_t) : 0);
  const size_t o_goff = take(G * E * sizeof(int32_t));
  const size_t o_tor = take(E * R * sizeof(int32_t));
  const size_t o_xe = take(E * R * d * h->es);
  const size_t o_h = take(E * R * F * h->es);
  const size_t o_ye = take(E * R * d * h->es);
  const bool train_tc = train && cfg->dtype == SWITCH_BF16 && tc_shape_ok((int)F, (int)d) && tc_shape_ok((int)d, (int)F);
  const size_t o_bdye = take(train ? E * R * d * sizeof(float) : 0);
  const size_t o_bdh = take(train && !train_tc ? E * R * F * sizeof(float) : 0);   // CUDA-core path only
  const size_t o_bdxe = take(train && !train_tc ? E * R * d * sizeof(float) : 0);
  const size_t o_bdg = take(train ? N * sizeof(float) : 0);
  const size_t o_bdz = take(train ? N * E * sizeof(float) : 0);
  // token chunks of the router's weight-gradient sums: ~256 tokens each, the partials
  // [nsplit, E, d] kept under 64 M floats
  const size_t part_cap = (size_t)64 << 20;
  size_t nsplit = N > 0 ? (N + 255) / 256 : 1;
  const size_t cap = std::max<size_t>(1, part_cap / std::max<size_t>(1, E * d));
  if (nsplit > cap) nsplit = cap;
  // tensor-core router products: E % 64 == 0 and kc-row token chunks (kc a multiple of 64
  // dividing N) with at most 64 chunks and partials [ntc, 2E, d] under the same cap
  size_t kc = 0, ntc = 0;
  if (train_tc && E % 64 == 0 && N > 0) {
    const size_t cands[] = {256, 512, 1024, 2048, 4096, 8192, 16384, 32768, 65536, 131072, 128, 64};
    for (size_t k : cands) {
      if (k > N || N % k != 0) continue;
      const size_t ns = N / k;
      if (ns <= 64 && ns * 2 * E * d <= part_cap) {
        kc = k;
        ntc = ns;
        break;
      }
    }
  }
  const size_t part_floats = std::max(nsplit * E * d, ntc * 2 * E * d);
  const size_t o_bpart = take(train ? part_floats * sizeof(float) : 0);
  const size_t o_dzp = take(ntc ? N * 3 * E * 2 : 0);
  const size_t o_wp = take(ntc ? 3 * E * d * 2 : 0);
  const size_t o_rowsk = take(ntc ? (ntc + 1) * sizeof(int32_t) : 0);
  const size_t o_dye16 = take(train_tc ? E * R * d * 2 : 0);
  const size_t o_dh16 = take(train_tc ? E * R * F * 2 : 0);
  const size_t o_dxe16 = take(train_tc ? E * R * d * 2 : 0);
  const size_t Rpad = (R + 63) / 64 * 64;
  const size_t o_rows2 = take(train_tc ? 2 * E * sizeof(int32_t) : 0);
  const size_t cw2 = std::max(1 + E * ((std::max(d, F) + 255) / 256),
                              std::max(1 + ntc * ((2 * E + 255) / 256), 1 + (N + 255) / 256));
  const size_t o_cnt2 = take(train_tc ? cw2 * sizeof(uint32_t) : 0);
  h->ws_bytes = off;
  if (cudaMalloc(&h->ws, h->ws_bytes) != cudaSuccess) {
    cudaGetLastError();
    delete h;
    return SWITCH_ERR_OOM;
  }
  h->err = reinterpret_cast<uint32_t*>(h->ws + o_err);
  h->logits = reinterpret_cast<float*>(h->ws + o_logits);
  h->tile_hist = reinterpret_cast<int32_t*>(h->ws + o_hist);
  h->tile_P = reinterpret_cast<float*>(h->ws + o_tP);
  h->tile_Z = reinterpret_cast<float*>(h->ws + o_tZ);
  h->tile_hist2 = reinterpret_cast<int32_t*>(h->ws + o_hist2);
  h->tile_base2 = reinterpret_cast<int32_t*>(h->ws + o_base2);
  h->tile_base = reinterpret_cast<int32_t*>(h->ws + o_base);
  h->group_off = reinterpret_cast<int32_t*>(h->ws + o_goff);
  h->tok_of_row = reinterpret_cast<int32_t*>(h->ws + o_tor);
  h->wsplit = h->ws + o_wsplit;
  h->xchg = xchg_bytes ? h->ws + o_xchg : nullptr;
  h->scan_partial = reinterpret_cast<float*>(h->ws + o_part);
  h->ffn_counters = reinterpret_cast<uint32_t*>(h->ws + o_fcnt);
  h->ffn_counter_words = (int)ffn_words;
  h->scan_counter = h->err + 1;
  h->xe = h->ws + o_xe;
  h->hbuf = h->ws + o_h;
  h->ye = h->ws + o_ye;
  h->bw_dye = reinterpret_cast<float*>(h->ws + o_bdye);
  h->bw_dh = reinterpret_cast<float*>(h->ws + o_bdh);
  h->bw_dxe = reinterpret_cast<float*>(h->ws + o_bdxe);
  h->bw_dg = reinterpret_cast<float*>(h->ws + o_bdg);
  h->bw_dz = reinterpret_cast<float*>(h->ws + o_bdz);
  h->bw_part = reinterpret_cast<float*>(h->ws + o_bpart);
  h->bw_nsplit = (int)nsplit;
  h->bw_ntc = (int)ntc;
  h->bw_kc = (int)kc;
  h->bw_dzp = ntc ? h->ws + o_dzp : nullptr;
  h->bw_Wp = ntc ? h->ws + o_wp : nullptr;
  h->bw_rows_k = ntc ? reinterpret_cast<int32_t*>(h->ws + o_rowsk) : nullptr;
  h->bw_tc = train_tc;
  h->bw_dye16 = train_tc ? h->ws + o_dye16 : nullptr;
  h->bw_dh16 = train_tc ? h->ws + o_dh16 : nullptr;
  h->bw_dxe16 = train_tc ? h->ws + o_dxe16 : nullptr;
  h->bw_Rpad = (int)Rpad;
  h->bw_rows_d = reinterpret_cast<int32_t*>(h->ws + o_rows2);
  h->bw_rows_F = h->bw_rows_d + E;
  h->bw_counters = reinterpret_cast<uint32_t*>(h->ws + o_cnt2);
  h->bw_counter_words = (int)cw2;
  if (cudaMemset(h->ws, 0, h->ws_bytes) != cudaSuccess) {
    cudaFree(h->ws);
    delete h;
    return SWITCH_ERR_CUDA;
  }
  h->have_events = true;
  for (int i = 0; i < 6; ++i)
    if (cudaEventCreate(&h->ev[i]) != cudaSuccess) h->have_events = false;
  *out = h;
  return SWITCH_OK;
}

static void host_path_free(HostPath* p) {
  if (!p) return;
  if (p->cin) cudaStreamSynchronize(p->cin);
  if (p->cout) cudaStreamSynchronize(p->cout);
  cudaEvent_t* evs[3] = {p->in_done, p->fwd_done, p->out_done};
  for (int i = 0; i < p->n_events; ++i) cudaEventDestroy(evs[i / 2][i % 2]);
  if (p->cin) cudaStreamDestroy(p->cin);
  if (p->cout) cudaStreamDestroy(p->cout);
  if (p->stage) cudaFree(p->stage);
  delete p;
}

switch_status switch_destroy(switch_handle h) {
  if (!h) return SWITCH_ERR_INVALID_ARG;
  host_path_free(h->hp);
  if (h->have_events)
    for (int i = 0; i < 6; ++i) cudaEventDestroy(h->ev[i]);
  const cudaError_t e = cudaFree(h->ws);
  delete h;
  return e == cudaSuccess ? SWITCH_OK : SWITCH_ERR_CUDA;
}

static switch_status route_args(switch_handle h, const void* x, const float* Wr, const float* br,
                                const switch_route_out* out, RouteArgs* a) {
  if (!h || !route_out_ok(out, h ? h->N : 0, h && top2_of(&h->cfg))) return SWITCH_ERR_INVALID_ARG;
  // Wr may be NULL only for the tensor-core router with prepared weights
  if (!Wr && !(h->cfg.dtype == SWITCH_BF16 && h->wsplit_ready)) return SWITCH_ERR_INVALID_ARG;
  if (Wr && h->cfg.dtype == SWITCH_BF16 && h->N > 0) h->wsplit_ready = true;  // this call splits Wr
  if (h->N > 0 && !x) return SWITCH_ERR_INVALID_ARG;
  if (x && !aligned16(x)) return SWITCH_ERR_INVALID_ARG;
  const switch_config& c = h->cfg;
  const bool want_logits = (c.flags & SWITCH_FLAG_WRITE_LOGITS) && out->logits;
  const bool want_probs = (c.flags & SWITCH_FLAG_WRITE_PROBS) && out->probs;
  a->x = x;
  a->Wr = Wr;
  a->br = br;
  a->G = c.G;
  a->T = c.T;
  a->d = c.d_model;
  a->E = c.E;
  a->C = h->C;
  a->R = h->R;
  a->x_bf16 = c.dtype == SWITCH_BF16;
  a->alpha = c.alpha;
  a->debug = (c.flags & SWITCH_FLAG_DEBUG_BOUNDS) != 0;
  a->slots = true;
  a->logits = want_logits ? out->logits : h->logits;
  // training: the backward needs the logits, so the tensor-core router writes them too
  a->logits_out = want_logits ? out->logits : (training_of(&c) ? h->logits : nullptr);
  a->wsplit = h->wsplit;
  a->xchg = h->xchg;
  a->tile_hist = h->tile_hist;
  a->tile_P = h->tile_P;
  a->tile_Z = h->tile_Z;
  a->tile_base = h->tile_base;
  a->group_off = h->group_off;
  a->tok_of_row = h->tok_of_row;
  a->scan_partial = h->scan_partial;
  a->scan_counter = h->scan_counter;
  a->err = h->err;
  a->max_ctas = h->route_ctas;
  a->expert = out->expert;
  a->slot = out->slot;
  a->keep = out->keep;
  a->gate = out->gate;
  a->row = out->row;
  a->raw = out->raw_count;
  a->accepted = out->accepted_count;
  a->P = out->P;
  a->balance = out->balance;
  a->aux_g = out->aux_loss_per_group;
  a->aux = out->aux_loss;
  a->expert_rows = out->expert_rows;
  a->probs = want_probs ? out->probs : nullptr;
  a->z_g = out->z_loss_per_group;
  a->z = out->z_loss;
  a->top2 = top2_of(&c);
  if (a->top2) {
    a->expert2 = out->expert2;
    a->slot2 = out->slot2;
    a->keep2 = out->keep2;
    a->gate2 = out->gate2;
    a->row2 = out->row2;
    a->raw2 = out->raw2_count;
    a->accepted2 = out->accepted2_count;
    a->tile_hist2 = h->tile_hist2;
    a->tile_base2 = h->tile_base2;
  }
  return SWITCH_OK;
}

switch_status switch_route(switch_handle h, const void* x, const float* Wr, const float* br,
                           const switch_route_out* out, void* stream) {
  RouteArgs a{};
  const switch_status st = route_args(h, x, Wr, br, out, &a);
  if (st != SWITCH_OK) return st;
  return launched(launch_route(a, (cudaStream_t)stream), h);
}

switch_status switch_prepare_router(switch_handle h, const float* Wr, void* stream) {
  if (!h || !Wr) return SWITCH_ERR_INVALID_ARG;
  if (h->cfg.dtype != SWITCH_BF16) return SWITCH_ERR_UNSUPPORTED;
  if (launch_router_split(Wr, h->wsplit, h->cfg.E, h->cfg.d_model, (cudaStream_t)stream) < 0) return SWITCH_ERR_CUDA;
  h->wsplit_ready = true;
  return SWITCH_OK;
}

switch_status switch_dispatch(switch_handle h, const void* x, const switch_route_out* r, void* xe, void* stream) {
  if (!h || !route_out_ok(r, h->N, top2_of(&h->cfg)) || (h->R > 0 && !xe) || !aligned16(xe))
    return SWITCH_ERR_INVALID_ARG;
  if (h->N > 0 && (!x || !aligned16(x))) return SWITCH_ERR_INVALID_ARG;
  const bool two = top2_of(&h->cfg);
  return launched(launch_dispatch(x, xe, r->expert, r->row, two ? r->expert2 : nullptr, two ? r->row2 : nullptr,
                                  r->expert_rows, h->N, h->cfg.E, h->R, h->cfg.d_model * h->es, h->err,
                                  (cudaStream_t)stream),
                  h);
}

static bool use_tc_ffn(const switch_layer* h) {
  const switch_config& c = h->cfg;
  return c.dtype == SWITCH_BF16 && tc_shape_ok(c.d_ff, c.d_model) && tc_shape_ok(c.d_model, c.d_ff);
}

// Both FFN layers on the tensor cores (one persistent kernel).  combine: write y in
// token order (gate * expert output, + x_residual) instead of ye.
static switch_status run_ffn_tc(switch_handle h, const void* xe, const void* W1, const void* b1, const void* W2,
                                const void* b2, const int32_t* rows, void* out, bool combine,
                                const switch_route_out* r, const void* resid, cudaStream_t s, bool pdl) {
  const switch_config& c = h->cfg;
  FfnLaunch L{};
  L.xe = xe;
  L.W1 = W1;
  L.b1 = b1;
  L.W2 = W2;
  L.b2 = b2;
  L.h = h->hbuf;
  L.out = out;
  L.expert_rows = rows;
  L.combine = combine;
  L.tok_of_row = h->tok_of_row;
  L.gate = r ? r->gate : nullptr;
  L.resid = resid;
  L.counters = h->ffn_counters;
  L.err = h->err;
  L.E = c.E;
  L.R = h->R;
  L.d = c.d_model;
  L.F = c.d_ff;
  L.stall = (c.flags & SWITCH_FLAG_TEST_STALL) != 0;
  L.max_ctas = h->ffn_ctas;
  // training keeps h for the backward
  L.discard_h = training_of(&c) ? 0 : (c.flags & SWITCH_FLAG_TEST_DISCARD) ? 2 : 1;
  const int n = launch_ffn_tc(L, s, pdl);
  if (n < 0) return SWITCH_ERR_CUDA;
  h->last_launches += n;
  return SWITCH_OK;
}

// Both FFN layers on CUDA cores (float32, or widths the tensor-core tiles do not take).
static switch_status run_ffn_simt(switch_handle h, const void* xe, const void* W1, const void* b1, const void* W2,
                                  const void* b2, const int32_t* rows, void* ye, cudaStream_t s, int ev_mid,
                                  bool pdl) {
  const switch_config& c = h->cfg;
  const int E = c.E, R = h->R, d = c.d_model, F = c.d_ff;
  const bool bf16 = c.dtype == SWITCH_BF16;
  int n = launch_grouped_linear_simt(xe, W1, b1, h->hbuf, rows, E, R, F, d, true, bf16, s, pdl);
  if (n < 0) return SWITCH_ERR_CUDA;
  h->last_launches += n;
  if (ev_mid >= 0) cudaEventRecord(h->ev[ev_mid], s);
  n = launch_grouped_linear_simt(h->hbuf, W2, b2, ye, rows, E, R, d, F, false, bf16, s, ev_mid < 0);
  if (n < 0) return SWITCH_ERR_CUDA;
  h->last_launches += n;
  return SWITCH_OK;
}

switch_status switch_expert_ffn(switch_handle h, const void* xe, const void* W1, const void* b1, const void* W2,
                                const void* b2, const int32_t* expert_rows, void* ye, void* stream) {
  if (!h || !W1 || !W2 || !expert_rows) return SWITCH_ERR_INVALID_ARG;
  if (h->R > 0 && (!xe || !ye)) return SWITCH_ERR_INVALID_ARG;
  if (!aligned16(xe) || !aligned16(W1) || !aligned16(W2) || !aligned16(ye)) return SWITCH_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  if (use_tc_ffn(h)) {
    if (h->R == 0) return SWITCH_OK;
    if (cudaMemsetAsync(h->ffn_counters, 0, (size_t)h->ffn_counter_words * sizeof(uint32_t), s) != cudaSuccess)
      return SWITCH_ERR_CUDA;
    return run_ffn_tc(h, xe, W1, b1, W2, b2, expert_rows, ye, false, nullptr, nullptr, s, false);
  }
  return run_ffn_simt(h, xe, W1, b1, W2, b2, expert_rows, ye, s, -1, false);
}

static switch_status combine_impl(switch_handle h, const void* ye, const switch_route_out* r, const void* x_residual,
                                  void* y, cudaStream_t s, bool pdl) {
  const bool two = h && top2_of(&h->cfg);
  if (!h || !route_out_ok(r, h->N, two) || (h->R > 0 && !ye) || (h->N > 0 && !y) || !aligned16(ye) ||
      !aligned16(y))
    return SWITCH_ERR_INVALID_ARG;
  if (x_residual && !aligned16(x_residual)) return SWITCH_ERR_INVALID_ARG;
  return launched(launch_combine(ye, r->expert, r->row, r->gate, two ? r->expert2 : nullptr,
                                 two ? r->row2 : nullptr, two ? r->gate2 : nullptr, x_residual, y, h->N,
                                 h->cfg.d_model, h->cfg.E, h->R, h->cfg.dtype == SWITCH_BF16, h->err, s, pdl),
                  h);
}

switch_status switch_combine(switch_handle h, const void* ye, const switch_route_out* r, const void* x_residual,
                             void* y, void* stream) {
  return combine_impl(h, ye, r, x_residual, y, (cudaStream_t)stream, false);
}

switch_status switch_forward(switch_handle h, const void* x, const float* Wr, const float* br, const void* W1,
                             const void* b1, const void* W2, const void* b2, const switch_route_out* r,
                             const void* x_residual, void* y, void* stream) {
  if (!h || !W1 || !W2 || (h->N > 0 && !y) || !aligned16(y) || !aligned16(W1) || !aligned16(W2)) return SWITCH_ERR_INVALID_ARG;
  if (x_residual && !aligned16(x_residual)) return SWITCH_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  const bool prof = (h->cfg.flags & SWITCH_FLAG_PROFILE) && h->have_events;
  h->last_launches = 0;
  if (prof) cudaEventRecord(h->ev[0], s);
  // Consecutive kernels of the call start as programmatic dependents of their
  // predecessor (their prologues overlap its tail); with per-stage events in between
  // (SWITCH_FLAG_PROFILE) every launch is an ordinary one.
  RouteArgs a{};
  switch_status st = route_args(h, x, Wr, br, r, &a);
  if (st != SWITCH_OK) return st;
  if (a.top2 || training_of(&h->cfg)) {
    // top-2: routing with its slots, one dispatch pass for both choices, the FFN into ye,
    // and a combine that adds the two weighted outputs per token.  Training (top-1 or
    // top-2) takes the same unfused path, so xe, h and ye stay in the workspace for the
    // backward.
    a.slots = true;
    st = launched(launch_route(a, s), h);
    if (st != SWITCH_OK) return st;
    if (prof) cudaEventRecord(h->ev[1], s);
    st = launched(launch_dispatch(x, h->xe, r->expert, r->row, a.top2 ? r->expert2 : nullptr,
                                  a.top2 ? r->row2 : nullptr, r->expert_rows, h->N, h->cfg.E, h->R,
                                  h->cfg.d_model * h->es, h->err, s),
                  h);
    if (st != SWITCH_OK) return st;
    if (prof) cudaEventRecord(h->ev[2], s);
    if (use_tc_ffn(h)) {
      if (h->R > 0) {
        if (cudaMemsetAsync(h->ffn_counters, 0, (size_t)h->ffn_counter_words * sizeof(uint32_t), s) != cudaSuccess)
          return SWITCH_ERR_CUDA;
        st = run_ffn_tc(h, h->xe, W1, b1, W2, b2, r->expert_rows, h->ye, false, nullptr, nullptr, s, false);
        if (st != SWITCH_OK) return st;
      }
      if (prof) cudaEventRecord(h->ev[3], s);
    } else {
      st = run_ffn_simt(h, h->xe, W1, b1, W2, b2, r->expert_rows, h->ye, s, prof ? 3 : -1, !prof);
      if (st != SWITCH_OK) return st;
    }
    if (prof) cudaEventRecord(h->ev[4], s);
    st = combine_impl(h, h->ye, r, x_residual, y, s, false);
    if (st != SWITCH_OK) return st;
    if (prof) cudaEventRecord(h->ev[5], s);
    return SWITCH_OK;
  }
  a.slots = false;  // the dispatch pass below turns ranks into slots
  st = launched(launch_route(a, s), h);
  if (st != SWITCH_OK) return st;
  if (prof) cudaEventRecord(h->ev[1], s);
  const bool tc = use_tc_ffn(h);
  // With the tensor-core FFN the combine happens in its epilogue: the dispatch pass
  // writes the dropped tokens' rows of y and clears the FFN's scheduler counters.
  st = launched(launch_dispatch_slots(x, h->xe, a, tc ? y : nullptr, tc ? x_residual : nullptr,
                                      tc ? h->ffn_counters : nullptr, tc ? h->ffn_counter_words : 0, s, !prof),
                h);
  if (st != SWITCH_OK) return st;
  if (prof) cudaEventRecord(h->ev[2], s);
  if (tc) {
    if (h->R > 0) {
      st = run_ffn_tc(h, h->xe, W1, b1, W2, b2, r->expert_rows, y, true, r, x_residual, s, !prof);
      if (st != SWITCH_OK) return st;
    }
    if (prof) {
      cudaEventRecord(h->ev[3], s);
      cudaEventRecord(h->ev[4], s);
    }
  } else {
    st = run_ffn_simt(h, h->xe, W1, b1, W2, b2, r->expert_rows, h->ye, s, prof ? 3 : -1, !prof);
    if (st != SWITCH_OK) return st;
    if (prof) cudaEventRecord(h->ev[4], s);
    st = combine_impl(h, h->ye, r, x_residual, y, s, !prof);
    if (st != SWITCH_OK) return st;
  }
  if (prof) cudaEventRecord(h->ev[5], s);
  return SWITCH_OK;
}

static switch_status host_path_init(switch_handle h) {
  if (h->hp) return h->hp->ok ? SWITCH_OK : SWITCH_ERR_CUDA;
  HostPath* p = new (std::nothrow) HostPath();
  if (!p) return SWITCH_ERR_OOM;
  h->hp = p;
  p->act_bytes = (size_t)h->N * h->cfg.d_model * h->es;
  p->slot_stride = round_up(p->act_bytes, 256);
  if (cudaStreamCreateWithFlags(&p->cin, cudaStreamNonBlocking) != cudaSuccess ||
      cudaStreamCreateWithFlags(&p->cout, cudaStreamNonBlocking) != cudaSuccess)
    return SWITCH_ERR_CUDA;
  cudaEvent_t* evs[3] = {p->in_done, p->fwd_done, p->out_done};
  for (int i = 0; i < 6; ++i) {
    if (cudaEventCreateWithFlags(&evs[i / 2][i % 2], cudaEventDisableTiming) != cudaSuccess) return SWITCH_ERR_CUDA;
    p->n_events = i + 1;
  }
  if (cudaMalloc(&p->stage, 4 * p->slot_stride + 2 * 256) != cudaSuccess) {
    cudaGetLastError();
    p->stage = nullptr;
    return SWITCH_ERR_OOM;
  }
  p->ok = true;
  return SWITCH_OK;
}

switch_status switch_forward_host(switch_handle h, const void* x_host, const float* Wr, const float* br,
                                  const void* W1, const void* b1, const void* W2, const void* b2,
                                  const switch_route_out* r, int residual, void* y_host, float* aux_loss_host,
                                  void* done_event, void* stream) {
  if (!h || !r || (h->N > 0 && (!x_host || !y_host))) return SWITCH_ERR_INVALID_ARG;
  switch_status st = host_path_init(h);
  if (st != SWITCH_OK) return st;
  HostPath* p = h->hp;
  cudaStream_t s = (cudaStream_t)stream;
  const int k = (int)(p->calls & 1u);
  uint8_t* xs = p->stage + (size_t)k * p->slot_stride;
  uint8_t* ys = p->stage + (size_t)(2 + k) * p->slot_stride;
  float* as = reinterpret_cast<float*>(p->stage + 4 * p->slot_stride + (size_t)k * 256);
  const bool reuse = p->calls >= 2;  // slot k was used by the call before the previous one
  // copy in: after the layer of that call has read x from slot k
  if (reuse && cudaStreamWaitEvent(p->cin, p->fwd_done[k], 0) != cudaSuccess) return SWITCH_ERR_CUDA;
  // In four pieces (of at least 1 MiB): single host-to-device copies from page-locked memory
  // ran at 10-30 GB/s (12.6 MB) and 36-42 GB/s (100 MB) on some B300 hosts, where two to eight
  // pieces reached 53-55 GB/s; many small pieces (<= 4 MiB) slowed the copies down when the
  // copy out ran at the same time.
  const size_t piece = std::max<size_t>((size_t)1 << 20, ((p->act_bytes + 3) / 4 + 4095) / 4096 * 4096);
  for (size_t off = 0; off < p->act_bytes; off += piece)
    if (cudaMemcpyAsync(xs + off, static_cast<const uint8_t*>(x_host) + off, std::min(piece, p->act_bytes - off),
                        cudaMemcpyHostToDevice, p->cin) != cudaSuccess)
      return SWITCH_ERR_CUDA;
  if (cudaEventRecord(p->in_done[k], p->cin) != cudaSuccess) return SWITCH_ERR_CUDA;
  // the layer: after its input has landed and the copy out of that call has read y
  if (cudaStreamWaitEvent(s, p->in_done[k], 0) != cudaSuccess) return SWITCH_ERR_CUDA;
  if (reuse && cudaStreamWaitEvent(s, p->out_done[k], 0) != cudaSuccess) return SWITCH_ERR_CUDA;
  ++p->calls;
  st = switch_forward(h, xs, Wr, br, W1, b1, W2, b2, r, residual ? xs : nullptr, ys, stream);
  if (st != SWITCH_OK) return st;
  if (cudaMemcpyAsync(as, r->aux_loss, sizeof(float), cudaMemcpyDeviceToDevice, s) != cudaSuccess ||
      cudaEventRecord(p->fwd_done[k], s) != cudaSuccess)
    return SWITCH_ERR_CUDA;
  // copy out
  if (cudaStreamWaitEvent(p->cout, p->fwd_done[k], 0) != cudaSuccess) return SWITCH_ERR_CUDA;
  if (p->act_bytes && cudaMemcpyAsync(y_host, ys, p->act_bytes, cudaMemcpyDeviceToHost, p->cout) != cudaSuccess)
    return SWITCH_ERR_CUDA;
  if (aux_loss_host &&
      cudaMemcpyAsync(aux_loss_host, as, sizeof(float), cudaMemcpyDeviceToHost, p->cout) != cudaSuccess)
    return SWITCH_ERR_CUDA;
  if (cudaEventRecord(p->out_done[k], p->cout) != cudaSuccess) return SWITCH_ERR_CUDA;
  if (done_event) {
    if (cudaEventRecord((cudaEvent_t)done_event, p->cout) != cudaSuccess) return SWITCH_ERR_CUDA;
  } else if (cudaStreamWaitEvent(s, p->out_done[k], 0) != cudaSuccess) {
    return SWITCH_ERR_CUDA;
  }
  return SWITCH_OK;
}

switch_status switch_backward(switch_handle h, const void* x, const float* Wr, const void* W1, const void* W2,
                              const switch_route_out* r, const void* dy, float w_aux, float w_z, int residual,
                              float* dx, float* dWr, float* dbr, float* dW1, float* db1, float* dW2, float* db2,
                              void* stream) {
  if (!h || !Wr || !W1 || !W2 || !dWr || !dW1 || !dW2) return SWITCH_ERR_INVALID_ARG;
  if (!training_of(&h->cfg) || top2_of(&h->cfg)) return SWITCH_ERR_UNSUPPORTED;
  if (!route_out_ok(r, h->N)) return SWITCH_ERR_INVALID_ARG;
  if (h->N > 0 && (!x || !dy || !dx)) return SWITCH_ERR_INVALID_ARG;
  const switch_config& c = h->cfg;
  BackwardArgs a{};
  a.G = c.G;
  a.T = c.T;
  a.E = c.E;
  a.R = h->R;
  a.d = c.d_model;
  a.F = c.d_ff;
  a.bf16 = c.dtype == SWITCH_BF16;
  a.alpha = c.alpha;
  a.w_aux = w_aux;
  a.w_z = w_z;
  a.residual = residual != 0;
  a.x = x;
  a.dy = dy;
  a.Wr = Wr;
  a.W1 = W1;
  a.W2 = W2;
  a.xe = h->xe;
  a.h = h->hbuf;
  a.ye = h->ye;
  a.logits = ((c.flags & SWITCH_FLAG_WRITE_LOGITS) && r->logits) ? r->logits : h->logits;
  a.expert = r->expert;
  a.row = r->row;
  a.gate = r->gate;
  a.raw = r->raw_count;
  a.expert_rows = r->expert_rows;
  a.dx = dx;
  a.dWr = dWr;
  a.dbr = dbr;
  a.dW1 = dW1;
  a.db1 = db1;
  a.dW2 = dW2;
  a.db2 = db2;
  a.dye = h->bw_dye;
  a.dh = h->bw_dh;
  a.dxe = h->bw_dxe;
  a.dg = h->bw_dg;
  a.dz = h->bw_dz;
  a.tc = h->bw_tc;
  a.dye16 = h->bw_dye16;
  a.dh16 = h->bw_dh16;
  a.dxe16 = h->bw_dxe16;
  a.counters = h->ffn_counters;
  a.counter_words = h->ffn_counter_words;
  a.err = h->err;
  a.Rpad = h->bw_Rpad;
  a.rows_d = h->bw_rows_d;
  a.rows_F = h->bw_rows_F;
  a.counters2 = h->bw_counters;
  a.counter2_words = h->bw_counter_words;
  a.part = h->bw_part;
  a.nsplit = h->bw_nsplit;
  a.ntc = h->bw_ntc;
  a.kc = h->bw_kc;
  a.dzp = h->bw_dzp;
  a.Wp = h->bw_Wp;
  a.rows_k = h->bw_rows_k;
  h->last_launches = 0;
  return launched(launch_backward(a, (cudaStream_t)stream), h);
}

static switch_status read_error_word(switch_handle h, cudaStream_t s) {
  uint32_t word = 0;
  if (cudaMemcpyAsync(&word, h->err, sizeof(word), cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return SWITCH_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return SWITCH_ERR_CUDA;
  if (word) {
    if (cudaMemsetAsync(h->err, 0, sizeof(uint32_t), s) != cudaSuccess) return SWITCH_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return SWITCH_ERR_CUDA;
    return (word & ERR_TIMEOUT) ? SWITCH_ERR_DEVICE_TIMEOUT : SWITCH_ERR_DEVICE_BOUNDS;
  }
  return SWITCH_OK;
}

switch_status switch_get_stats(switch_handle h, const switch_route_out* r, void* stream, float* aux_loss_host,
                               int32_t* raw_host, int32_t* accepted_host, int64_t* dropped_host) {
  if (!h || !route_out_ok(r, h->N)) return SWITCH_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  const size_t GE = (size_t)h->cfg.G * h->cfg.E;
  if (cudaStreamSynchronize(s) != cudaSuccess) return SWITCH_ERR_CUDA;
  if (aux_loss_host && cudaMemcpy(aux_loss_host, r->aux_loss, sizeof(float), cudaMemcpyDeviceToHost) != cudaSuccess)
    return SWITCH_ERR_CUDA;
  if (raw_host && cudaMemcpy(raw_host, r->raw_count, GE * sizeof(int32_t), cudaMemcpyDeviceToHost) != cudaSuccess)
    return SWITCH_ERR_CUDA;
  int32_t* acc = accepted_host;
  int32_t* tmp = nullptr;
  if (!acc && dropped_host) {
    tmp = (int32_t*)malloc(GE * sizeof(int32_t));
    if (!tmp) return SWITCH_ERR_OOM;
    acc = tmp;
  }
  if (acc && cudaMemcpy(acc, r->accepted_count, GE * sizeof(int32_t), cudaMemcpyDeviceToHost) != cudaSuccess) {
    free(tmp);
    return SWITCH_ERR_CUDA;
  }
  if (dropped_host) {
    int64_t kept = 0;
    for (size_t i = 0; i < GE; ++i) kept += acc[i];
    *dropped_host = (int64_t)h->N - kept;
  }
  free(tmp);
  return read_error_word(h, s);
}

switch_status switch_sync_status(switch_handle h, void* stream) {
  if (!h) return SWITCH_ERR_INVALID_ARG;
  return read_error_word(h, (cudaStream_t)stream);
}

switch_status switch_stage_ms(switch_handle h, float* ms, int n) {
  if (!h || !ms || n < 5) return SWITCH_ERR_INVALID_ARG;
  if (!(h->cfg.flags & SWITCH_FLAG_PROFILE) || !h->have_events) return SWITCH_ERR_UNSUPPORTED;
  if (cudaEventSynchronize(h->ev[5]) != cudaSuccess) return SWITCH_ERR_CUDA;
  for (int i = 0; i < 5; ++i)
    if (cudaEventElapsedTime(&ms[i], h->ev[i], h->ev[i + 1]) != cudaSuccess) return SWITCH_ERR_CUDA;
  return SWITCH_OK;
}

int switch_last_launch_count(switch_handle h) { return h ? h->last_launches : -1; }

switch_status switch_set_sm_budget(switch_handle h, int route_ctas, int ffn_ctas) {
  if (!h || route_ctas < 0 || ffn_ctas < 0) return SWITCH_ERR_INVALID_ARG;
  h->route_ctas = route_ctas;
  h->ffn_ctas = ffn_ctas;
  return SWITCH_OK;
}

switch_status switch_ep_regroup(const void* src, void* dst, const int32_t* counts, int32_t* rows_out, int W, int El,
                                int R, int row_bytes, int inverse, void* stream) {
  if (W < 1 || El < 1 || R < 0 || row_bytes <= 0 || row_bytes % 16 != 0 || !counts) return SWITCH_ERR_INVALID_ARG;
  if ((long long)W * El * R >= (1ll << 31)) return SWITCH_ERR_INVALID_ARG;
  if ((long long)W * El * R > 0 && (!src || !dst || !aligned16(src) || !aligned16(dst))) return SWITCH_ERR_INVALID_ARG;
  if (inverse && rows_out) return SWITCH_ERR_INVALID_ARG;
  return launch_ep_regroup(src, dst, counts, rows_out, W, El, R, row_bytes, inverse != 0, (cudaStream_t)stream) < 0
             ? SWITCH_ERR_CUDA
             : SWITCH_OK;
}

}  // extern "C"

// ---------------------------------------------------------------- routing without a handle
// switch_route_static keeps everything the routing kernels need between them (the split
// router weights, per-tile statistics, scan state, the error word) in this one fixed
// device array instead of a workspace from switch_create.  Every GPU that loads the
// library holds it until the process exits.
namespace {

constexpr size_t STATIC_ROUTE_SCRATCH_BYTES = (size_t)32 << 20;  // 32 MiB
__device__ __align__(256) uint8_t g_static_route_scratch[STATIC_ROUTE_SCRATCH_BYTES];

// Device address of the array in the current device's context.  Looked up on every call:
// the name is only a host-side stand-in and must never be handed to a kernel, and after a
// context reset (cudaDeviceReset) the array lives at a new address, so a cached one could
// go stale.  Once the library's device code is loaded on the device the lookup is a host
// table read.
void* static_route_scratch() {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_static_route_scratch) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  return p;
}

}  // namespace

extern "C" switch_status switch_route_static(const switch_config* cfg, const void* x, const float* Wr,
                                             const float* br, const switch_route_out* out, void* stream) {
  if (!config_ok(cfg) || !Wr) return SWITCH_ERR_INVALID_ARG;
  if (top2_of(cfg)) return SWITCH_ERR_UNSUPPORTED;  // top-2 routing needs a handle's logits buffer
  const int N = cfg->G * cfg->T;
  if (!route_out_ok(out, N)) return SWITCH_ERR_INVALID_ARG;
  if (N > 0 && !x) return SWITCH_ERR_INVALID_ARG;
  if (x && !aligned16(x)) return SWITCH_ERR_INVALID_ARG;
  const int C = (int)capacity_of(cfg);
  const int Ceff = C < cfg->T ? C : cfg->T;
  const int R = cfg->G * Ceff;
  const int nT = (cfg->T + ROUTE_TILE - 1) / ROUTE_TILE;
  const size_t E = cfg->E, G = cfg->G, d = cfg->d_model;
  const bool bf16 = cfg->dtype == SWITCH_BF16;
  // layout of the scratch, as in a handle's workspace (route part only)
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = round_up(off + bytes, 256);
    return o;
  };
  const size_t o_err = take(sizeof(uint32_t) * 4);  // [0] error word, [1] scan counter
  const size_t o_logits = take(bf16 ? 0 : (size_t)N * E * sizeof(float));
  const size_t o_wsplit = take(bf16 ? router_tc_wsplit_bytes(cfg->E, cfg->d_model) : 0);
  const size_t o_hist = take(G * nT * E * sizeof(int32_t));
  const size_t o_tP = take(G * nT * E * sizeof(float));
  const size_t o_tZ = take(G * nT * sizeof(float));
  const size_t o_base = take(G * nT * E * sizeof(int32_t));
  const size_t o_goff = take(G * E * sizeof(int32_t));
  const size_t o_tor = take(E * (size_t)R * sizeof(int32_t));
  const size_t o_part = take(G * (size_t)route_scan_blocks(cfg->E) * sizeof(float));
  if (off > STATIC_ROUTE_SCRATCH_BYTES) return SWITCH_ERR_UNSUPPORTED;  // needs more than 32 MiB
  (void)d;
  uint8_t* ws = static_cast<uint8_t*>(static_route_scratch());
  if (!ws) return SWITCH_ERR_CUDA;
  cudaStream_t s = (cudaStream_t)stream;
  // the error word and the scan's block counter must start at zero; everything else is
  // written by the kernels before it is read
  if (cudaMemsetAsync(ws + o_err, 0, sizeof(uint32_t) * 4, s) != cudaSuccess) return SWITCH_ERR_CUDA;
  const bool want_logits = (cfg->flags & SWITCH_FLAG_WRITE_LOGITS) && out->logits;
  const bool want_probs = (cfg->flags & SWITCH_FLAG_WRITE_PROBS) && out->probs;
  RouteArgs a{};
  a.x = x;
  a.Wr = Wr;
  a.br = br;
  a.G = cfg->G;
  a.T = cfg->T;
  a.d = cfg->d_model;
  a.E = cfg->E;
  a.C = C;
  a.R = R;
  a.x_bf16 = bf16;
  a.alpha = cfg->alpha;
  a.debug = (cfg->flags & SWITCH_FLAG_DEBUG_BOUNDS) != 0;
  a.slots = true;
  a.logits = want_logits ? out->logits : reinterpret_cast<float*>(ws + o_logits);
  a.logits_out = want_logits ? out->logits : nullptr;
  a.wsplit = ws + o_wsplit;
  a.tile_hist = reinterpret_cast<int32_t*>(ws + o_hist);
  a.tile_P = reinterpret_cast<float*>(ws + o_tP);
  a.tile_Z = reinterpret_cast<float*>(ws + o_tZ);
  a.tile_base = reinterpret_cast<int32_t*>(ws + o_base);
  a.group_off = reinterpret_cast<int32_t*>(ws + o_goff);
  a.tok_of_row = reinterpret_cast<int32_t*>(ws + o_tor);
  a.scan_partial = reinterpret_cast<float*>(ws + o_part);
  a.scan_counter = reinterpret_cast<uint32_t*>(ws + o_err) + 1;
  a.err = reinterpret_cast<uint32_t*>(ws + o_err);
  a.expert = out->expert;
  a.slot = out->slot;
  a.keep = out->keep;
  a.gate = out->gate;
  a.row = out->row;
  a.raw = out->raw_count;
  a.accepted = out->accepted_count;
  a.P = out->P;
  a.balance = out->balance;
  a.aux_g = out->aux_loss_per_group;
  a.aux = out->aux_loss;
  a.expert_rows = out->expert_rows;
  a.probs = want_probs ? out->probs : nullptr;
  a.z_g = out->z_loss_per_group;
  a.z = out->z_loss;
  return launch_route(a, s) < 0 ? SWITCH_ERR_CUDA : SWITCH_OK;
}
