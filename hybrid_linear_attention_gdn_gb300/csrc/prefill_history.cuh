// Types shared by the prefill kernels (prefill.cu) and the single-launch
// mixed step (prefill_tc32.cu), and the conv-history work of a prefill.
#pragma once
#include "gdn_common.cuh"

namespace gdn {
namespace pfx {

constexpr int kMaxW = 8;
constexpr int kCkGroup = 4;  // checkpoints per history-kernel thread

struct PrefillArgs {
  float* ssm;
  void* conv;
  int32_t num_slots;
  float* ck_ssm;
  void* ck_conv;
  int32_t ck_num_slots;
  const float* conv_w;
  const float* A_log;
  const float* dt_bias;
  const int32_t* slot_ids;
  const int32_t* cu_seqlens;
  const int64_t* start_pos;
  int32_t n_seq;
  int64_t total;
  const int32_t* ckpt_ids;
  int32_t max_ckpt;
  int32_t ckpt_block;
  const void* qkv;
  const void* a;
  const void* b;
  void* out;
  uint32_t* err;
  // workspace (fp32)
  float* ws_q;     // [total][hk][dk]  q^ (scaled by dk^-1/2)
  float* ws_k;     // [total][hk][dk]  k^
  float* ws_v;     // [total][hv][dv]
  float* ws_g;     // [total][hv]      log decay g
  float* ws_beta;  // [total][hv]
  int32_t hk, hv, dk, dv, W, C, G;
};

// The caller's tensors and the workspace of a prefill as checked views
// (extents in elements).
template <typename Tact, typename Tconv>
struct PrefillViews {
  View<float, 0> ssm, ck_ssm, ws_q, ws_k, ws_v, ws_g, ws_beta;
  View<Tconv, 0> conv, ck_conv;
  View<const float, 0> conv_w, A_log, dt_bias;
  View<const int32_t, 0> slot_ids, cu_seqlens, ckpt_ids;
  View<const int64_t, 0> start_pos;
  View<const Tact, 0> qkv, a, b;
  View<Tact, 0> out;
  __device__ __forceinline__ explicit PrefillViews(const PrefillArgs& g) {
    const long long slot_n = (long long)g.hv * g.dv * g.dk, hist_n = (long long)(g.W - 1) * g.C;
    ssm = GDN_GV(g.ssm, g.num_slots * slot_n);
    ck_ssm = GDN_GV(g.ck_ssm, g.ck_num_slots * slot_n);
    conv = GDN_GV(reinterpret_cast<Tconv*>(g.conv), g.num_slots * hist_n);
    ck_conv = GDN_GV(reinterpret_cast<Tconv*>(g.ck_conv), g.ck_num_slots * hist_n);
    ws_q = GDN_GV(g.ws_q, g.total * g.hk * g.dk);
    ws_k = GDN_GV(g.ws_k, g.total * g.hk * g.dk);
    ws_v = GDN_GV(g.ws_v, g.total * g.hv * g.dv);
    ws_g = GDN_GV(g.ws_g, g.total * g.hv);
    ws_beta = GDN_GV(g.ws_beta, g.total * g.hv);
    conv_w = GDN_GV(g.conv_w, (long long)g.C * g.W);
    A_log = GDN_GV(g.A_log, g.hv);
    dt_bias = GDN_GV(g.dt_bias, g.hv);
    slot_ids = GDN_GV(g.slot_ids, g.n_seq);
    cu_seqlens = GDN_GV(g.cu_seqlens, g.n_seq + 1);
    ckpt_ids = GDN_GV(g.ckpt_ids, (long long)g.n_seq * g.max_ckpt);
    start_pos = GDN_GV(g.start_pos, g.n_seq);
    qkv = GDN_GV(reinterpret_cast<const Tact*>(g.qkv), g.total * g.C);
    a = GDN_GV(reinterpret_cast<const Tact*>(g.a), g.total * g.hv);
    b = GDN_GV(reinterpret_cast<const Tact*>(g.b), g.total * g.hv);
    out = GDN_GV(reinterpret_cast<Tact*>(g.out), g.total * g.hv * g.dv);
  }
};

// The conv histories of sequence n, channel c: the checkpoints of group
// grp (kCkGroup of them) and, for group 0, the working slot's final history.
// A checkpoint's history is the raw input of the 3 (W - 1) positions before
// its block boundary; the final one that of the sequence's last positions;
// positions before the sequence start come from the old history, which the
// caller guarantees no prefill kernel still has to read.
template <typename Tact, typename Tconv>
__device__ __forceinline__ void history_channel(const PrefillArgs& a, const int n, const int grp, const int c) {
  if (c >= a.C) return;
  const PrefillViews<Tact, Tconv> g(a);
  const int32_t slot = g.slot_ids[n];
  if (slot_class(slot, a.num_slots)) return;
  const int64_t t0 = g.cu_seqlens[n], len = (int64_t)g.cu_seqlens[n + 1] - t0;
  const int64_t p0 = g.start_pos[n], p1 = p0 + len;
  if (t0 < 0 || len < 0 || t0 + len > a.total || p0 < 0) return;
  const auto hist = g.conv + (size_t)slot * (a.W - 1) * a.C;
  const auto qkv = g.qkv;
  // Group 0 owns the working slot's history: it reads the old rows before
  // writing the new ones, and only its first checkpoint can reach back into
  // them (later checkpoints lie at least one 64-token block further on).
  float old[kMaxW];
#pragma unroll
  for (int j = 0; j < kMaxW - 1; ++j)
    if (j < a.W - 1) old[j] = grp == 0 ? to_f32(hist[(size_t)j * a.C + c]) : 0.f;
  // raw input at sequence-relative index m (negative: the old history)
  auto raw = [&](int64_t m) -> float {
    if (m >= 0) return to_f32(qkv[(t0 + m) * a.C + c]);
    float v = 0.f;
#pragma unroll
    for (int j = 0; j < kMaxW - 1; ++j)
      if (j == a.W - 1 + m) v = old[j];
    return v;
  };
  const int64_t blk = a.ckpt_block;
#pragma unroll
  for (int k = 0; k < kCkGroup; ++k) {
    const int idx = grp * kCkGroup + k;
    const int64_t P = (p0 / blk + 1 + idx) * blk;
    if (idx >= a.max_ckpt || P > p1) break;
    const int32_t cid = g.ckpt_ids[(size_t)n * a.max_ckpt + idx];
    const int cc = slot_class(cid, a.ck_num_slots);
    if (cc == 2 && c == 0) report(a.err, GDN_DEV_ERR_SLOT_OOB);
    if (cc) continue;
    const auto ch = g.ck_conv + (size_t)cid * (a.W - 1) * a.C;
    for (int j = 0; j < a.W - 1; ++j)
      ch[(size_t)j * a.C + c] = from_f32<Tconv>(raw(P - p0 - (a.W - 1) + j));
  }
  if (grp != 0) return;
  float nw[kMaxW];
#pragma unroll
  for (int j = 0; j < kMaxW - 1; ++j)
    if (j < a.W - 1) nw[j] = raw(len - (a.W - 1) + j);
#pragma unroll
  for (int j = 0; j < kMaxW - 1; ++j)
    if (j < a.W - 1) hist[(size_t)j * a.C + c] = from_f32<Tconv>(nw[j]);
}


}  // namespace pfx
}  // namespace gdn
