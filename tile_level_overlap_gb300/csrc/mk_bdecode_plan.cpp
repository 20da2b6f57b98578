// Host plan of the tensor-core batched decode queue (see mk_bdecode.h).
// Every GEMM row tile is released once, by the last of its K chunks to
// arrive; every (sequence, kv head) attention group once, by the last of its
// splits.  Waiters count those releases.  Where a consumer's K chunk reads
// only some producer tiles, it waits on just those (barriers partitioned
// along the dependency dimension, "Lecture 112: Production Megakernels for
// Real-World Inference", Key takeaways): a down-projection chunk of 1024
// SwiGLU columns on the 16 gate/up row tiles that write them, an
// O-projection chunk of 1024 attention-output columns on the kv groups whose
// heads those are, a QKV or gate/up chunk of 1024 hidden features on the 8
// down or O row tiles that write them.  The RMSNorm-folded projections scale
// their outputs by 1 / rms of the whole row, which needs every producer row
// tile: their epilogue runs in the last chunk of the row tile to arrive, when
// all chunks have passed their waits, so together they have covered every
// producer tile.
#include <algorithm>
#include <cstring>
#include <map>

#include "mk_bdecode.h"
#include "mk_plan.h"

namespace mk {

namespace {

Instr bd_make(uint8_t op, int layer, uint32_t a0, uint32_t a1, uint16_t a2 = 0) {
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

void bd_wait(Instr& in, uint32_t bar, uint32_t target, uint16_t n = 1) {
  in.wait_bar = bar;
  in.wait_target = target;
  in.wait_n = n;
  in.wait_stride = 1;
}

uint32_t chunks(int K) { return (uint32_t)((K + BD_KC - 1) / BD_KC); }

}  // namespace

int build_bdecode(const mk_model_cfg& c, int max_batch, int max_ctx, int n_sms, BdPlan* out,
                  std::string* why) {
  auto bad = [&](int code, const char* msg) {
    if (why) *why = msg;
    return code;
  };
  if (c.n_layers < 1 || c.n_layers > MAX_LAYERS || c.hidden < 64 || c.n_q_heads < 1 ||
      c.n_kv_heads < 1 || c.ffn < 64 || c.vocab < 1 || max_ctx < 2)
    return bad(MK_ERR_INVALID_ARG, "bad model dimensions or context");
  if (c.n_q_heads % c.n_kv_heads) return bad(MK_ERR_INVALID_ARG, "n_q_heads % n_kv_heads != 0");
  if (max_batch < 1 || max_batch > BD_NMAX)
    return bad(MK_ERR_UNSUPPORTED, "tensor-core decode takes 1..32 sequences");
  if (c.head_dim != 64 && c.head_dim != 128)
    return bad(MK_ERR_UNSUPPORTED, "tensor-core decode head_dim must be 64 or 128");
  const int rep = c.n_q_heads / c.n_kv_heads;
  // the tensor-core attention scores pair q row g (hi) with row g + rep (lo)
  // by a lane xor of 4 * rep: rep must be a power of two
  if (rep != 1 && rep != 2 && rep != 4)
    return bad(MK_ERR_UNSUPPORTED, "tensor-core decode takes 1, 2 or 4 q heads per kv head");
  const int qd = c.n_q_heads * c.head_dim, kd = c.n_kv_heads * c.head_dim;
  if (c.hidden % BD_M || qd % BD_M || kd % BD_M || c.ffn % (BD_M / 2) || c.hidden % BD_BK ||
      c.ffn % BD_BK || qd % BD_BK)
    return bad(MK_ERR_UNSUPPORTED,
               "tensor-core decode needs hidden, n_q*d, n_kv*d % 128 == 0 and ffn % 64 == 0");
  auto chunk_ok = [](int K) { return K <= BD_KC ? true : K % BD_KC == 0; };
  if (!chunk_ok(c.hidden) || !chunk_ok(qd) || !chunk_ok(c.ffn))
    return bad(MK_ERR_UNSUPPORTED, "K dimensions above 1024 must be multiples of 1024");
  BdPlan& bp = *out;
  bp = BdPlan();
  bp.cfg = c;
  bp.max_batch = max_batch;
  bp.max_ctx = max_ctx;
  bp.nb = max_batch <= 16 ? 16 : 32;
  // Attention splits per (sequence, kv head): four.  Measured on the
  // Llama-3-8B shape at batch 8 (64 groups over 152 SMs): 2 splits 8.31 ms,
  // 4 splits 6.96 ms, 8 splits 7.41 ms per step (fewer splits lengthen the
  // phase's critical tile; more add combine work and per-tile overhead).
  (void)n_sms;
  bp.nsplit = 4;
  bp.rep = rep;
  bp.qkv_rows = qd + 2 * kd;
  bp.n_rg = (max_batch + BD_RG - 1) / BD_RG;
  bp.n_qkv_m = (uint32_t)(bp.qkv_rows / BD_M);
  bp.n_o_m = (uint32_t)(c.hidden / BD_M);
  bp.n_gu_m = (uint32_t)(c.ffn / (BD_M / 2));
  bp.n_down_m = (uint32_t)(c.hidden / BD_M);
  bp.n_lm_m = (uint32_t)((c.vocab + BD_M - 1) / BD_M);
  bp.c_h = chunks(c.hidden);
  // O in 512-column chunks (one kv group of heads at rep 4, head_dim 128):
  // each chunk waits on fewer attention groups and starts sooner
  bp.c_q = qd > BD_KC ? (uint32_t)(qd / (BD_KC / 2)) : chunks(qd);
  bp.c_f = chunks(c.ffn);
  // gate/up reads the whole hidden row for each of its 224 (Llama-3-8B) row
  // tiles: 2048-column chunks halve its tile count (448 tiles, about three
  // rounds over the SMs) and the per-tile overhead
  bp.c_g = (c.hidden > BD_KC && c.hidden % (2 * BD_KC) == 0) ? (uint32_t)(c.hidden / (2 * BD_KC)) : bp.c_h;
  // QKV's 48 (Llama-3-8B) row tiles: 512-column chunks give 384 tiles, about
  // two and a half rounds, instead of 192 (one round and a quarter)
  bp.c_k = c.hidden > BD_KC ? (uint32_t)(c.hidden / (BD_KC / 2)) : bp.c_h;

  const int L = c.n_layers, nkv = c.n_kv_heads;
  // kv groups per 1024-column chunk of the attention output, gate/up row
  // tiles (64 SwiGLU columns each) per 1024-column chunk of the FFN
  const uint32_t g_per_c = qd <= BD_KC ? (uint32_t)nkv : (uint32_t)((BD_KC / 2) / (rep * c.head_dim));
  const uint32_t gu_per_c = c.ffn <= BD_KC ? bp.n_gu_m : (uint32_t)(BD_KC / (BD_M / 2));
  // O / down row tiles (128 hidden features each) per 1024-feature chunk
  const uint32_t h_per_c = c.hidden <= BD_KC ? bp.n_down_m : (uint32_t)(BD_KC / BD_M);
  // QKV row tiles per kv group: at head_dim 128 every 128-row tile holds one
  // head (q, k or v) of one group, and an attention group waits on just its
  // rep + 2 tiles; at head_dim 64 a k or v tile spans two groups, and every
  // group waits on the whole projection
  const bool qkv_by_group = c.head_dim == BD_M;
  const uint32_t ng = qkv_by_group ? (uint32_t)nkv : 1u;
  const uint32_t qkv_per_g = qkv_by_group ? (uint32_t)rep + 2u : bp.n_qkv_m;
  const uint32_t mq = (uint32_t)(qd / BD_M), mk = (uint32_t)(kd / BD_M);
  auto qkv_group = [&](uint32_t m) -> uint32_t {
    if (!qkv_by_group) return 0;
    if (m < mq) return m / (uint32_t)rep;
    return m < mq + mk ? m - mq : m - mq - mk;
  };
  // emission order of the QKV row tiles: group by group (its q heads, its k,
  // its v), so the first groups' attention can start first
  std::vector<uint32_t> qkv_order;
  if (qkv_by_group) {
    for (uint32_t g = 0; g < (uint32_t)nkv; ++g) {
      for (uint32_t r = 0; r < (uint32_t)rep; ++r) qkv_order.push_back(g * rep + r);
      qkv_order.push_back(mq + g);
      qkv_order.push_back(mq + mk + g);
    }
  } else {
    for (uint32_t m = 0; m < bp.n_qkv_m; ++m) qkv_order.push_back(m);
  }
  BdBars& b = bp.bl;
  b.norm1 = 0;
  b.qkv = b.norm1 + L;                     // [L][ng]
  b.attn = b.qkv + L * ng;                 // [L][n_kv]
  b.o = b.attn + L * nkv;                  // [L][c_h]
  b.norm2 = b.o + L * bp.c_h;
  b.gu = b.norm2 + L;                      // [L][c_f]
  b.down = b.gu + L * bp.c_f;              // [L][c_h]
  b.normf = b.down + L * bp.c_h;
  b.lm = b.normf + 1;
  b.total = b.lm + 1;

  std::vector<Instr>& q = bp.queue;
  auto begin = [&]() { return (uint32_t)q.size(); };
  auto end = [&](uint32_t s) {
    if (q.size() > s) bp.perop.push_back({s, (uint32_t)q.size() - s});
  };
  // wait(ch): first barrier, count and per-barrier target of chunk ch;
  // rel(m): the barrier row tile m releases
  struct Wait {
    uint32_t bar, target;
    uint16_t n;
  };
  auto gemm_rows = [&](uint8_t op, int l, const std::vector<uint32_t>& rows, uint32_t nc, auto&& wait,
                       auto&& rel) {
    const uint32_t s = begin();
    for (uint32_t m : rows)
      for (uint32_t ch = 0; ch < nc; ++ch) {
        Instr in = bd_make(op, l, m, ch);
        const Wait w = wait(ch);
        bd_wait(in, w.bar, w.target, w.n);
        in.rel_bar = rel(m);
        q.push_back(in);
      }
    end(s);
  };
  auto gemm = [&](uint8_t op, int l, uint32_t nm, uint32_t nc, auto&& wait, auto&& rel) {
    std::vector<uint32_t> rows(nm);
    for (uint32_t m = 0; m < nm; ++m) rows[m] = m;
    gemm_rows(op, l, rows, nc, wait, rel);
  };
  // chunk by chunk (every row tile of chunk 0, then of chunk 1, ...): for an
  // operator whose chunks become ready one after another, so that a tile
  // popped early is one whose inputs come early, rather than a later chunk's
  // tile that would hold its SM while it waits
  auto gemm_by_chunk = [&](uint8_t op, int l, uint32_t nm, uint32_t nc, auto&& wait, auto&& rel) {
    const uint32_t s = begin();
    for (uint32_t ch = 0; ch < nc; ++ch)
      for (uint32_t m = 0; m < nm; ++m) {
        Instr in = bd_make(op, l, m, ch);
        const Wait w = wait(ch);
        bd_wait(in, w.bar, w.target, w.n);
        in.rel_bar = rel(m);
        q.push_back(in);
      }
    end(s);
  };
  auto all = [](uint32_t bar, uint32_t target) { return [=](uint32_t) { return Wait{bar, target, 1}; }; };
  auto one = [](uint32_t bar) { return [=](uint32_t) { return bar; }; };
  auto norm = [&](uint8_t op, int l, uint32_t wbar, uint32_t wtarget, uint32_t rbar) {
    const uint32_t s = begin();
    for (int r = 0; r < bp.n_rg; ++r) {
      Instr in = bd_make(op, l, (uint32_t)r, 0);
      if (wbar != NO_BAR) bd_wait(in, wbar, wtarget);
      in.rel_bar = rbar;
      q.push_back(in);
    }
    end(s);
  };
  // layer 0's input norm is its own instruction (the embedding rows); every
  // later norm is folded into the O / down epilogues (see mk_bdecode.h)
  norm(BD_NORM1, 0, NO_BAR, 0, b.norm1);
  for (int l = 0; l < L; ++l) {
    auto qkv_rel = [&](uint32_t m) { return b.qkv + l * ng + qkv_group(m); };
    if (l == 0)
      gemm_rows(BD_QKV, l, qkv_order, bp.c_k, all(b.norm1, (uint32_t)bp.n_rg), qkv_rel);
    else
      gemm_rows(BD_QKV, l, qkv_order, bp.c_k,
                [&](uint32_t ch) {
                  // the 1024-feature down chunk that holds this chunk's columns
                  return Wait{b.down + (l - 1) * bp.c_h + ch * bp.c_h / bp.c_k, h_per_c, 1};
                },
                qkv_rel);
    {
      // kv group by kv group (every sequence of a group, then the next
      // group): the first groups finish first, and the O chunks that read
      // only their heads start while the later groups are still running
      const uint32_t s = begin();
      for (int g = 0; g < nkv; ++g)
        for (int bb = 0; bb < max_batch; ++bb)
          for (int sp = 0; sp < bp.nsplit; ++sp) {
            Instr in = bd_make(BD_ATTN, l, (uint32_t)bb, (uint32_t)g, (uint16_t)sp);
            bd_wait(in, b.qkv + l * ng + (qkv_by_group ? (uint32_t)g : 0u), qkv_per_g);
            in.rel_bar = b.attn + l * nkv + g;
            q.push_back(in);
          }
      end(s);
    }
    // O chunk ch: the kv groups of its 1024 attention-output columns, every
    // sequence of each
    gemm_by_chunk(BD_O, l, bp.n_o_m, bp.c_q,
         [&](uint32_t ch) {
           return Wait{b.attn + l * nkv + ch * g_per_c, (uint32_t)max_batch, (uint16_t)g_per_c};
         },
         [&](uint32_t m) { return b.o + l * bp.c_h + m / h_per_c; });
    // gate/up chunk ch: the O row tiles of its 1024 hidden features; row
    // tile m writes SwiGLU columns [64 m, 64 m + 64)
    gemm(BD_GU, l, bp.n_gu_m, bp.c_g,
         [&](uint32_t ch) {
           const uint32_t r = bp.c_h / bp.c_g;  // 1024-feature O chunks per gate/up chunk
           return Wait{b.o + l * bp.c_h + ch * r, h_per_c, (uint16_t)r};
         },
         [&](uint32_t m) { return b.gu + l * bp.c_f + m / gu_per_c; });
    // down chunk ch: the gate/up row tiles of its 1024 SwiGLU columns
    gemm_by_chunk(BD_DOWN, l, bp.n_down_m, bp.c_f,
         [&](uint32_t ch) { return Wait{b.gu + l * bp.c_f + ch, gu_per_c, 1}; },
         [&](uint32_t m) { return b.down + l * bp.c_h + m / h_per_c; });
  }
  // the LM head is not split over K: every down row tile of the last layer
  gemm(BD_LM, L - 1, bp.n_lm_m, 1,
       [&](uint32_t) { return Wait{b.down + (L - 1) * bp.c_h, h_per_c, (uint16_t)bp.c_h}; },
       one(b.lm));
  return MK_OK;
}

// Sequential check of a queue order: every wait is satisfied when reached and
// every barrier ends with exactly the releases its waiters expect.  A GEMM row
// tile releases once when its last chunk arrives; an attention group once
// when its last split arrives.
int simulate_bdecode(const BdPlan& bp, const std::vector<Instr>& q, std::string* why) {
  std::vector<uint32_t> cnt(bp.bl.total, 0);
  std::map<uint64_t, uint32_t> arrived;
  auto group_size = [&](const Instr& in) -> uint32_t {
    switch (in.op) {
      case BD_QKV: return bp.c_k;
      case BD_GU: return bp.c_g;
      case BD_O: return bp.c_q;
      case BD_DOWN: return bp.c_f;
      case BD_ATTN: return (uint32_t)bp.nsplit;
      default: return 1;
    }
  };
  for (size_t i = 0; i < q.size(); ++i) {
    const Instr& in = q[i];
    if (in.op < BD_NORM1 || in.op > BD_LM) {
      if (why) *why = "unknown batched-decode opcode at " + std::to_string(i);
      return MK_ERR_INVALID_ARG;
    }
    if (in.wait_bar != NO_BAR) {
      for (uint32_t k = 0; k < in.wait_n; ++k) {
        const uint32_t wb = in.wait_bar + k * in.wait_stride;
        if (wb >= bp.bl.total || cnt[wb] < in.wait_target) {
          if (why) *why = "batched-decode instruction " + std::to_string(i) + " waits before its producers";
          return MK_ERR_INVALID_ARG;
        }
      }
    }
    if (in.rel_bar == NO_BAR) continue;
    const uint32_t gs = group_size(in);
    if (gs == 1) {
      cnt[in.rel_bar] += 1;
      continue;
    }
    const uint64_t key = ((uint64_t)in.op << 56) | ((uint64_t)in.layer << 40) |
                         (in.op == BD_ATTN ? ((uint64_t)in.a0 << 20 | in.a1) : (uint64_t)in.a0);
    if (++arrived[key] == gs) cnt[in.rel_bar] += 1;
  }
  for (size_t i = 0; i < q.size(); ++i) {
    const Instr& in = q[i];
    if (in.wait_bar == NO_BAR) continue;
    for (uint32_t k = 0; k < in.wait_n; ++k)
      if (cnt[in.wait_bar + k * in.wait_stride] != in.wait_target) {
        if (why) *why = "batched-decode barrier count mismatch at instruction " + std::to_string(i);
        return MK_ERR_INVALID_ARG;
      }
  }
  return MK_OK;
}

// A seeded random topological order of the queue (for schedule-invariance
// tests): repeatedly takes a random instruction whose wait is satisfied.
void random_order_bdecode(const BdPlan& bp, uint64_t seed, std::vector<Instr>* out) {
  const std::vector<Instr>& q = bp.queue;
  out->clear();
  std::vector<uint32_t> cnt(bp.bl.total, 0);
  std::vector<std::vector<uint32_t>> waiters(bp.bl.total);
  std::vector<uint32_t> ready, pending(q.size(), 0);  // pending: barriers not yet at target
  for (uint32_t i = 0; i < q.size(); ++i) {
    if (q[i].wait_bar == NO_BAR) {
      ready.push_back(i);
      continue;
    }
    pending[i] = q[i].wait_n;
    for (uint32_t k = 0; k < q[i].wait_n; ++k) waiters[q[i].wait_bar + k * q[i].wait_stride].push_back(i);
  }
  std::map<uint64_t, uint32_t> arrived;
  auto group_size = [&](const Instr& in) -> uint32_t {
    switch (in.op) {
      case BD_QKV: return bp.c_k;
      case BD_GU: return bp.c_g;
      case BD_O: return bp.c_q;
      case BD_DOWN: return bp.c_f;
      case BD_ATTN: return (uint32_t)bp.nsplit;
      default: return 1;
    }
  };
  uint64_t x = seed * 0x9E3779B97F4A7C15ull + 1;
  while (!ready.empty()) {
    x ^= x << 13; x ^= x >> 7; x ^= x << 17;
    const size_t k = (size_t)(x % ready.size());
    const uint32_t i = ready[k];
    ready[k] = ready.back();
    ready.pop_back();
    const Instr& in = q[i];
    out->push_back(in);
    if (in.rel_bar == NO_BAR) continue;
    const uint32_t gs = group_size(in);
    bool fire = gs == 1;
    if (!fire) {
      const uint64_t key = ((uint64_t)in.op << 56) | ((uint64_t)in.layer << 40) |
                           (in.op == BD_ATTN ? ((uint64_t)in.a0 << 20 | in.a1) : (uint64_t)in.a0);
      fire = ++arrived[key] == gs;
    }
    if (!fire) continue;
    const uint32_t c = ++cnt[in.rel_bar];
    for (uint32_t w : waiters[in.rel_bar])
      if (q[w].wait_target == c && --pending[w] == 0) ready.push_back(w);
  }
}

}  // namespace mk
