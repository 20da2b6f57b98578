// Host plan builder.  Turns a model shape into the tile DAG of one decode step,
// emitted as a topological instruction queue with per-tile barrier counters.
//
// Following the MegaOps Abstract, each consumer waits on the tiles of the
// intermediate tensor it reads: attention of kv group g waits only on the QKV
// row tiles of g's heads; every other dependency of a decode step is a
// reduction over the whole hidden vector (the RMSNorm before QKV / gate-up and
// the input dimension of O / down), so those barriers count every producer
// tile of the operator ("Lecture 112: Production Megakernels for Real-World
// Inference", Key takeaways: barriers held as tensors).  The counters define
// the DAG that the host simulator and the random topological orders check;
// on the device the decode interpreter enforces the same dependencies through
// the tag each element of an intermediate tensor carries (mk_device.cuh), a
// barrier tensor partitioned down to single elements.  Extents that depend on
// the batch or a sequence's cached length are expressions evaluated on the
// device, so the queue does not change with them (same source, symbolic
// shapes in S and P).
#include "mk_plan.h"

#include <algorithm>

#include "mk_variants.h"
#include <cstring>
#include <random>

namespace mk {

namespace {

int pow2_floor(int x) {
  int p = 1;
  while (p * 2 <= x) p *= 2;
  return p;
}

int rows_for(long target_bytes, long row_bytes, int cap) {
  long r = target_bytes / row_bytes;
  if (r < 1) r = 1;
  if (r > cap) r = cap;
  return pow2_floor((int)r);
}

uint32_t ceil_div(uint64_t a, uint64_t b) { return (uint32_t)((a + b - 1) / b); }

// Rows per tile such that an operator's tiles come in whole rounds over the
// SMs: about `target_bytes` per tile, rounded to a whole number of rounds of
// n_sms tiles (at least one), at most `cap` rows.  An operator that waits on an
// all-to-all input then starts with one tile per SM, which the operand ring has
// largely prefetched during the wait, instead of a ragged second round.
int rows_rounds(long total_rows, long row_bytes, long target_bytes, int n_sms, int cap) {
  const double rounds_f = (double)total_rows * row_bytes / ((double)n_sms * target_bytes);
  long rounds = (long)(rounds_f + 0.5);
  if (rounds < 1) rounds = 1;
  long r = (total_rows + rounds * n_sms - 1) / (rounds * n_sms);
  if (r < 1) r = 1;
  if (r > cap) r = cap;
  return (int)r;
}

Instr make(Op op, int layer, uint32_t a0, uint32_t a1, uint16_t a2 = 0) {
  Instr in;
  std::memset(&in, 0, sizeof(in));
  in.op = op;
  in.layer = (uint16_t)layer;
  in.a0 = a0;
  in.a1 = a1;
  in.a2 = a2;
  in.x_lo = NO_EXPR;
  in.x_hi = NO_EXPR;
  in.wait_bar = NO_BAR;
  in.rel_bar = NO_BAR;
  return in;
}

void set_wait(Instr& in, uint32_t bar, uint32_t target, uint16_t n = 1, uint16_t stride = 1) {
  in.wait_bar = bar;
  in.wait_target = target;
  in.wait_n = n;
  in.wait_stride = stride;
}

// Postfix expression helpers.  `depth` tracks the evaluation stack, which
// x_eval holds in X_STACK registers.
struct XBuild {
  std::vector<uint32_t> w;
  int sp = 0, depth = 0;
  XBuild& c(uint32_t v) { return push(xw(X_CONST, v)); }
  XBuild& op(uint32_t o) {
    if (o <= X_S) return push(xw(o));
    w.push_back(xw(o));
    if (o != X_POS) --sp;  // binary operators pop two, push one
    return *this;
  }
  XBuild& push(uint32_t word) {
    w.push_back(word);
    depth = ++sp > depth ? sp : depth;
    return *this;
  }
};

// Store an expression in its slot; false when it does not fit the slot's
// words or the evaluation stack.
bool put_expr(std::vector<uint32_t>& table, int slot, const XBuild& x) {
  if (x.w.size() >= (size_t)X_MAX_WORDS || x.depth > X_STACK) return false;
  for (size_t i = 0; i < x.w.size(); ++i) table[(size_t)slot * X_MAX_WORDS + i] = x.w[i];
  return true;
}

}  // namespace

int build_plan(const mk_model_cfg& c, int max_batch, int max_ctx, int n_sms, HostPlan* out,
               std::string* why) {
  auto bad = [&](int code, const char* msg) {
    if (why) *why = msg;
    return code;
  };
  if (c.n_layers < 1 || c.hidden < 8 || c.n_q_heads < 1 || c.n_kv_heads < 1 || c.head_dim < 2 ||
      c.ffn < 8 || c.vocab < 1)
    return bad(MK_ERR_INVALID_ARG, "model dimensions must be positive (n_layers >= 1)");
  if (c.n_q_heads % c.n_kv_heads) return bad(MK_ERR_INVALID_ARG, "n_q_heads % n_kv_heads != 0");
  if (!(c.rms_eps >= 0.f) || !(c.rope_theta > 0.f))
    return bad(MK_ERR_INVALID_ARG, "rms_eps must be >= 0 and rope_theta > 0");
  if (max_batch < 1 || max_ctx < 1) return bad(MK_ERR_INVALID_ARG, "max_batch, max_ctx >= 1");
  if (c.n_layers > MAX_LAYERS) return bad(MK_ERR_UNSUPPORTED, "more layers than the kernel holds");
  if (c.head_dim != 64 && c.head_dim != 128)
    return bad(MK_ERR_UNSUPPORTED, "head_dim must be 64 or 128");
  const int rep = c.n_q_heads / c.n_kv_heads;
  if (rep != 1 && rep != 2 && rep != 4 && rep != 8)
    return bad(MK_ERR_UNSUPPORTED, "query heads per kv head must be 1, 2, 4 or 8");
  const int qd = c.n_q_heads * c.head_dim;
  if (c.hidden % 8 || c.ffn % 8 || qd % 8)
    return bad(MK_ERR_UNSUPPORTED, "hidden, ffn and n_q_heads*head_dim must be multiples of 8");
  if (max_batch > BMAX_CC) return bad(MK_ERR_UNSUPPORTED, "batch above the CUDA-core decode limit");
  const int kmax = std::max(std::max(c.hidden, c.ffn), qd);
  static_assert(FAST_K_UNIT == 2048, "fast-path shapes assume 8 columns x 256 threads");
  const bool fast =
      has_fast_variant(c.hidden, c.ffn, c.n_q_heads, c.n_kv_heads, c.head_dim);
  // The generic path (batch > 1, or K outside the fast set) holds x[B][K] in
  // shared memory.
  if ((!fast || max_batch > 1) && (long)max_batch * kmax > XBUF_FLOATS)
    return bad(MK_ERR_UNSUPPORTED,
               "max_batch * max(K) exceeds the shared-memory activation buffer of the "
               "CUDA-core decode path");
  if ((long)c.head_dim * 2 > STAGE_BYTES || (long)kmax * 2 > STAGE_BYTES)
    return bad(MK_ERR_UNSUPPORTED, "a weight row does not fit one ring stage");

  HostPlan& hp = *out;
  hp = HostPlan();
  hp.cfg = c;
  hp.max_batch = max_batch;
  hp.max_ctx = max_ctx;
  hp.rep = rep;
  hp.qkv_rows = (c.n_q_heads + 2 * c.n_kv_heads) * c.head_dim;
  hp.fast_b1 = fast;

  const int L = c.n_layers, H = c.hidden, d = c.head_dim, F = c.ffn, nkv = c.n_kv_heads;
  if (n_sms <= 0) n_sms = DEFAULT_SMS;
  // Rows per tile: ~128-384 KB of weights per instruction amortises the
  // per-instruction handshakes; QKV tiles stay inside one head.  The down
  // projection takes the larger tiles (Llama-3-8B shape: two rounds of 14
  // rows instead of three of 9; 2.828 -> 2.804 ms per step measured).
  hp.r_qkv = std::min(rows_for(128 << 10, (long)H * 2, RMAX), d);
  hp.r_o = rows_rounds(H, (long)qd * 2, 256 << 10, n_sms, RMAX);
  hp.r_gu = rows_rounds(F, (long)H * 4, 256 << 10, n_sms, RMAX / 2);
  hp.r_down = rows_rounds(H, (long)F * 2, 384 << 10, n_sms, RMAX);
  hp.r_lm = rows_for(256 << 10, (long)H * 2, RMAX);
  hp.n_qkv_tiles = hp.qkv_rows / hp.r_qkv;
  hp.n_o_tiles = ceil_div(H, hp.r_o);
  hp.n_gu_tiles = ceil_div(F, hp.r_gu);
  hp.n_down_tiles = ceil_div(H, hp.r_down);
  hp.n_lm_tiles = ceil_div(c.vocab, hp.r_lm);

  // Split-KV partitions per (sequence, kv head): a fixed number of keys per
  // split (a model constant, keys_per_split), so which keys each partial
  // holds -- and with it every bit of the result -- depends only on the model
  // and the sequence's cached length, never on the device's SM count or the
  // plan's max_batch.  The queue holds ceil(max_ctx / KPS) splits per group;
  // splits past a sequence's keys are empty and cost one pop.
  hp.kps = keys_per_split(d);
  hp.split_max = SCORE_FLOATS / rep;
  if (hp.kps > hp.split_max) return bad(MK_ERR_UNSUPPORTED, "keys per split above the score buffer");
  const int ns = std::max(1, (int)ceil_div(max_ctx, hp.kps));
  hp.n_splits = ns;
  hp.n_comb = combine_slices(ns, rep, d);
  if (hp.n_splits > 0xffff || 2L * hp.n_splits * rep + rep > XBUF_FLOATS)
    return bad(MK_ERR_UNSUPPORTED, "max_ctx needs more split-KV partitions than the combine buffer holds");

  // Barrier tensor layout.
  BarLayout& bl = hp.bl;
  bl.qkv = 0;
  bl.split = bl.qkv + L * nkv;
  bl.attn = bl.split + L * max_batch * nkv;
  bl.o = bl.attn + L;
  bl.gu = bl.o + L;
  bl.down = bl.gu + L;
  bl.lm = bl.down + L;
  bl.total = bl.lm + 1;

  // Symbolic extents.  n = P[a0] + 1 keys; split a2 holds keys
  // [a2 * KPS, (a2 + 1) * KPS) clipped to n.
  hp.expr.assign((size_t)XS_COUNT * X_MAX_WORDS, 0);
  {
    XBuild lo;  // min(a2 * KPS, n)
    lo.op(X_ARG2).c(hp.kps).op(X_MUL).op(X_ARG0).op(X_POS).c(1).op(X_ADD).op(X_MIN);
    bool fits = put_expr(hp.expr, XS_ATTN_LO, lo);
    XBuild hi;  // min((a2 + 1) * KPS, n)
    hi.op(X_ARG2).c(1).op(X_ADD).c(hp.kps).op(X_MUL).op(X_ARG0).op(X_POS).c(1).op(X_ADD).op(X_MIN);
    fits = put_expr(hp.expr, XS_ATTN_HI, hi) && fits;
    XBuild live;  // B - a0
    live.op(X_B).op(X_ARG0).op(X_SUB);
    fits = put_expr(hp.expr, XS_SEQ_LIVE, live) && fits;
    if (!fits) return bad(MK_ERR_UNSUPPORTED, "extent expression exceeds the evaluator");
  }

  const uint32_t per_group = (uint32_t)(rep * d + 2 * d) / hp.r_qkv;
  auto group_of_row = [&](int row) {
    if (row < qd) return (row / d) / rep;
    if (row < qd + nkv * d) return (row - qd) / d;
    return (row - qd - nkv * d) / d;
  };

  std::vector<Instr>& q = hp.decode;
  q.clear();
  hp.perop_decode.clear();
  auto range_begin = [&]() { return (uint32_t)q.size(); };
  auto range_end = [&](uint32_t b) {
    if (q.size() > b) hp.perop_decode.push_back({b, (uint32_t)q.size() - b});
  };
  for (int l = 0; l < L; ++l) {
    uint32_t b0 = range_begin();
    for (int r = 0; r < hp.qkv_rows; r += hp.r_qkv) {
      Instr in = make(OP_QKV, l, r, hp.r_qkv);
      if (l > 0) set_wait(in, bl.down + l - 1, hp.n_down_tiles);
      in.rel_bar = bl.qkv + l * nkv + group_of_row(r);
      q.push_back(in);
    }
    range_end(b0);
    b0 = range_begin();
    // Split-KV attention, then the combine of each (sequence, kv head)
    // group.  Sliced (n_comb > 1): every split is an ordinary split and
    // n_comb combine instructions per group each wait on the group's splits
    // and combine a slice of its outputs.  Otherwise the group's last split
    // also combines the group (it waits on the other splits; a group's only
    // split combines its own partial).  Each group's last split follows the
    // layer's other splits (it holds keys only for contexts near max_ctx, and
    // an empty split among the others would push a split that holds keys into
    // a later round), and the combining instructions of a layer follow all its
    // splits, so the kernel-per-operator runner launches them as their own
    // operator.
    const bool sliced = ns > 1 && hp.n_comb > 1;
    const uint32_t n_comb = sliced ? (uint32_t)hp.n_comb : 1u;
    auto split_instr = [&](int b, int g, int s) {
      Instr in = make(OP_ATTN, l, b, g, (uint16_t)s);
      in.x_lo = XS_ATTN_LO;
      in.x_hi = XS_ATTN_HI;
      const uint32_t grp = ((uint32_t)l * max_batch + b) * nkv + g;
      if (s + 1 < ns || sliced) {
        set_wait(in, bl.qkv + l * nkv + g, per_group);
        in.rel_bar = bl.split + grp;
      } else {
        in.flags = IF_COMBINE;
        if (ns > 1) set_wait(in, bl.split + grp, (uint32_t)(ns - 1));
        else set_wait(in, bl.qkv + l * nkv + g, per_group);
        in.rel_bar = bl.attn + l;
      }
      q.push_back(in);
    };
    for (int b = 0; b < max_batch; ++b)
      for (int g = 0; g < nkv; ++g)
        for (int s = 0; s + 1 < ns; ++s) split_instr(b, g, s);
    if (sliced) {
      for (int b = 0; b < max_batch; ++b)
        for (int g = 0; g < nkv; ++g) split_instr(b, g, ns - 1);
    }
    range_end(b0);
    b0 = range_begin();
    for (int b = 0; b < max_batch; ++b)
      for (int g = 0; g < nkv; ++g) {
        if (!sliced) {
          split_instr(b, g, ns - 1);
          continue;
        }
        for (int c = 0; c < hp.n_comb; ++c) {
          Instr in = make(OP_ATTN, l, b, g, (uint16_t)c);
          in.flags = IF_COMBINE | IF_SLICE;
          set_wait(in, bl.split + ((uint32_t)l * max_batch + b) * nkv + g, (uint32_t)ns);
          in.rel_bar = bl.attn + l;
          q.push_back(in);
        }
      }
    range_end(b0);
    b0 = range_begin();
    for (int r = 0; r < H; r += hp.r_o) {
      Instr in = make(OP_O, l, r, std::min(hp.r_o, H - r));
      set_wait(in, bl.attn + l, (uint32_t)(max_batch * nkv) * n_comb);
      in.rel_bar = bl.o + l;
      q.push_back(in);
    }
    range_end(b0);
    b0 = range_begin();
    for (int r = 0; r < F; r += hp.r_gu) {
      Instr in = make(OP_GU, l, r, std::min(hp.r_gu, F - r));
      set_wait(in, bl.o + l, hp.n_o_tiles);
      in.rel_bar = bl.gu + l;
      q.push_back(in);
    }
    range_end(b0);
    b0 = range_begin();
    for (int r = 0; r < H; r += hp.r_down) {
      Instr in = make(OP_DOWN, l, r, std::min(hp.r_down, H - r));
      set_wait(in, bl.gu + l, hp.n_gu_tiles);
      in.rel_bar = bl.down + l;
      q.push_back(in);
    }
    range_end(b0);
  }
  uint32_t b0 = range_begin();
  for (int r = 0; r < c.vocab; r += hp.r_lm) {
    Instr in = make(OP_LM, L - 1, r, std::min(hp.r_lm, c.vocab - r));
    set_wait(in, bl.down + L - 1, hp.n_down_tiles);
    in.rel_bar = bl.lm;
    q.push_back(in);
  }
  range_end(b0);

  const uint64_t per_layer = (uint64_t)hp.qkv_rows * H + (uint64_t)H * qd + 3ull * F * H;
  hp.weight_bytes = 2 * (per_layer * L + (uint64_t)c.vocab * H);
  return MK_OK;
}

DecodeScratch decode_scratch(const HostPlan& hp) {
  const mk_model_cfg& c = hp.cfg;
  const size_t L = (size_t)c.n_layers, B = (size_t)hp.max_batch, H = (size_t)c.hidden;
  const size_t d = (size_t)c.head_dim, nkv = (size_t)c.n_kv_heads;
  const size_t w = sizeof(unsigned long long);  // one tagged word per element
  DecodeScratch x{};
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off += (bytes + 255) & ~(size_t)255;
    return o;
  };
  x.o_resid = take(w * (2 * L + 1) * B * H);
  x.o_qkv = take(w * L * B * hp.qkv_rows);
  x.o_part = take(w * L * B * nkv * hp.n_splits * hp.rep * (d + 2));
  x.o_attn = take(w * L * B * c.n_q_heads * d);
  x.o_act = take(w * L * B * c.ffn);
  x.tagged_end = off;
  x.o_bars = take(sizeof(uint32_t) * hp.bl.total);
  x.o_ctl = take(sizeof(uint32_t) * CTL_WORDS);
  x.zero_end = off;
  x.o_q = take(sizeof(Instr) * hp.decode.size());
  x.o_rope = take(sizeof(float2) * (size_t)hp.max_ctx * (d / 2));
  x.o_lw = take(sizeof(LayerW) * L);
  x.total = off;
  return x;
}

namespace {

// Apply `in`'s release to the counters; returns the barrier that received +1,
// or NO_BAR.
uint32_t apply_release(const Instr& in, std::vector<uint32_t>& cnt) {
  if (in.rel_bar == NO_BAR) return NO_BAR;
  cnt[in.rel_bar] += 1;
  return in.rel_bar;
}

}  // namespace

void random_topological(const HostPlan& hp, const std::vector<Instr>& q, uint64_t seed,
                        std::vector<Instr>* out) {
  const uint32_t nb = hp.bl.total;
  std::vector<uint32_t> cnt(nb, 0), target(nb, 0);
  std::vector<std::vector<uint32_t>> waiters(nb);
  std::vector<uint32_t> unmet(q.size(), 0);
  std::vector<uint32_t> ready;
  for (uint32_t i = 0; i < q.size(); ++i) {
    const Instr& in = q[i];
    if (in.wait_bar == NO_BAR || in.wait_n == 0) {
      ready.push_back(i);
      continue;
    }
    for (uint32_t k = 0; k < in.wait_n; ++k) {
      uint32_t b = in.wait_bar + k * in.wait_stride;
      waiters[b].push_back(i);
      target[b] = in.wait_target;
      unmet[i]++;
    }
  }
  std::mt19937_64 rng(seed);
  out->clear();
  out->reserve(q.size());
  while (!ready.empty()) {
    size_t pick = (size_t)(rng() % ready.size());
    uint32_t i = ready[pick];
    ready[pick] = ready.back();
    ready.pop_back();
    out->push_back(q[i]);
    uint32_t b = apply_release(q[i], cnt);
    if (b != NO_BAR && cnt[b] == target[b])
      for (uint32_t w : waiters[b])
        if (--unmet[w] == 0) ready.push_back(w);
  }
}

int simulate(const HostPlan& hp, const std::vector<Instr>& q, std::string* why) {
  std::vector<uint32_t> cnt(hp.bl.total, 0);
  for (size_t i = 0; i < q.size(); ++i) {
    const Instr& in = q[i];
    if (in.op == OP_NOP || in.op >= OP_COUNT) {
      if (why) *why = "unknown opcode at index " + std::to_string(i);
      return MK_ERR_INVALID_ARG;
    }
    if (in.wait_bar != NO_BAR)
      for (uint32_t k = 0; k < in.wait_n; ++k) {
        uint32_t b = in.wait_bar + k * in.wait_stride;
        if (b >= hp.bl.total || cnt[b] < in.wait_target) {
          if (why)
            *why = "instruction " + std::to_string(i) + " waits on barrier " + std::to_string(b) +
                   " before its producers ran";
          return MK_ERR_INVALID_ARG;
        }
      }
    apply_release(in, cnt);
  }
  for (size_t i = 0; i < q.size(); ++i) {
    const Instr& in = q[i];
    if (in.wait_bar == NO_BAR) continue;
    for (uint32_t k = 0; k < in.wait_n; ++k) {
      uint32_t b = in.wait_bar + k * in.wait_stride;
      if (cnt[b] != in.wait_target) {
        if (why)
          *why = "barrier " + std::to_string(b) + " receives " + std::to_string(cnt[b]) +
                 " releases but instruction " + std::to_string(i) + " expects " +
                 std::to_string(in.wait_target);
        return MK_ERR_INVALID_ARG;
      }
    }
  }
  return MK_OK;
}

}  // namespace mk
