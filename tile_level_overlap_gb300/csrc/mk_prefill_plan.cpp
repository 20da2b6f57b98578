// Host plan of the prefill queue: per layer, for 128-token blocks m,
//   NORM1(m) -> QKV(m, n) -> ATTN(m, g) -> O(m, n) -> NORM2(m) -> GU(m, n) -> DOWN(m, n)
// and the next layer's NORM1(m) waits only on DOWN(m, *) of block m.
// Attention of block m waits on the QKV tiles of blocks 0..m only (causal
// dependency), so early blocks flow into attention and the next layer while
// later blocks are still in their projections.
#include <algorithm>
#include <cstring>

#include "mk_plan.h"
#include "mk_prefill.h"

namespace mk {

namespace {

Instr pf_make(uint8_t op, int layer, uint32_t a0, uint32_t a1) {
  Instr in;
  std::memset(&in, 0, sizeof(in));
  in.op = op;
  in.layer = (uint16_t)layer;
  in.a0 = a0;
  in.a1 = a1;
  in.x_lo = PXS_BLOCK_LIVE;
  in.x_hi = NO_EXPR;
  in.wait_bar = NO_BAR;
  in.rel_bar = NO_BAR;
  return in;
}

}  // namespace

int build_prefill(const mk_model_cfg& c, int max_ctx, PrefillPlan* out, std::string* why) {
  auto bad = [&](int code, const char* msg) {
    if (why) *why = msg;
    return code;
  };
  if (c.n_layers < 1 || c.n_layers > MAX_LAYERS || c.hidden < 64 || c.n_q_heads < 1 ||
      c.n_kv_heads < 1 || c.ffn < 64 || c.vocab < 1 || max_ctx < 1)
    return bad(MK_ERR_INVALID_ARG, "bad model dimensions or context");
  if (c.n_q_heads % c.n_kv_heads) return bad(MK_ERR_INVALID_ARG, "n_q_heads % n_kv_heads != 0");
  if (c.head_dim != 64 && c.head_dim != 128)
    return bad(MK_ERR_UNSUPPORTED, "prefill head_dim must be 64 or 128");
  const int qd = c.n_q_heads * c.head_dim, kd = c.n_kv_heads * c.head_dim;
  if (c.hidden % PF_BN || c.ffn % PF_BN_GU || qd % 128 || kd % 128)
    return bad(MK_ERR_UNSUPPORTED,
               "prefill needs hidden % 256, ffn % 128 and head columns % 128 == 0");
  PrefillPlan& pp = *out;
  pp = PrefillPlan();
  pp.cfg = c;
  pp.max_ctx = max_ctx;
  pp.n_blocks = (max_ctx + PF_BM - 1) / PF_BM;
  pp.rep = c.n_q_heads / c.n_kv_heads;
  pp.qkv_rows = qd + 2 * kd;
  pp.bn_qkv = (qd % 256 == 0 && kd % 256 == 0) ? 256 : 128;
  pp.n_qkv_n = (uint32_t)(pp.qkv_rows / pp.bn_qkv);
  pp.n_o_n = (uint32_t)(c.hidden / PF_BN);
  pp.n_gu_n = (uint32_t)(c.ffn / PF_BN_GU);
  pp.n_down_n = (uint32_t)(c.hidden / PF_BN);
  pp.n_lm_n = (uint32_t)((c.vocab + PF_BN - 1) / PF_BN);

  const int L = c.n_layers, NB = pp.n_blocks, nkv = c.n_kv_heads;
  PfBars& b = pp.bl;
  const uint32_t per = (uint32_t)(L * NB);
  b.norm1 = 0;
  b.qkv = b.norm1 + per;
  b.attn = b.qkv + per;
  b.o = b.attn + per;
  b.norm2 = b.o + per;
  b.gu = b.norm2 + per;
  b.down = b.gu + per;
  b.normf = b.down + per;
  b.lm = b.normf + (uint32_t)NB;
  b.total = b.lm + (uint32_t)NB;
  auto bar = [&](uint32_t base, int l, int m) { return base + (uint32_t)(l * NB + m); };

  pp.expr.assign((size_t)PXS_COUNT * X_MAX_WORDS, 0);
  {
    uint32_t* e = &pp.expr[PXS_BLOCK_LIVE * X_MAX_WORDS];
    int i = 0;
    e[i++] = xw(X_S);
    e[i++] = xw(X_ARG0);
    e[i++] = xw(X_CONST, PF_BM);
    e[i++] = xw(X_MUL);
    e[i++] = xw(X_SUB);
  }

  std::vector<Instr>& q = pp.queue;
  // GEMM tiles go group by group of token blocks, and within a group weight
  // tile by weight tile, so the blocks of a group read each weight tile from
  // L2 right after the first of them brought it in.  Groups of up to
  // PF_BLOCK_GROUP blocks, and at least two groups: the first group's blocks
  // then run ahead into attention and the next layer while the second's are
  // in their projections.
  const int grp = std::max(1, std::min(PF_BLOCK_GROUP, NB / 2));
  auto grouped = [&](uint32_t nn, auto&& emit) {
    for (int mg = 0; mg < NB; mg += grp)
      for (uint32_t n = 0; n < nn; ++n)
        for (int m = mg; m < NB && m < mg + grp; ++m) emit(m, n);
  };
  auto begin = [&]() { return (uint32_t)q.size(); };
  auto end = [&](uint32_t s) {
    if (q.size() > s) pp.perop.push_back({s, (uint32_t)q.size() - s});
  };
  for (int l = 0; l < L; ++l) {
    uint32_t s = begin();
    for (int m = 0; m < NB; ++m) {
      Instr in = pf_make(PF_NORM1, l, m, 0);
      if (l > 0) {
        in.wait_bar = bar(b.down, l - 1, m);
        in.wait_target = pp.n_down_n;
        in.wait_n = 1;
        in.wait_stride = 1;
      }
      in.rel_bar = bar(b.norm1, l, m);
      q.push_back(in);
    }
    end(s);
    s = begin();
    grouped(pp.n_qkv_n, [&](int m, uint32_t n) {
      Instr in = pf_make(PF_QKV, l, m, n);
      in.wait_bar = bar(b.norm1, l, m);
      in.wait_target = 1;
      in.wait_n = 1;
      in.wait_stride = 1;
      in.rel_bar = bar(b.qkv, l, m);
      q.push_back(in);
    });
    end(s);
    s = begin();
    for (int m = 0; m < NB; ++m)
      for (int g = 0; g < nkv; ++g) {
        Instr in = pf_make(PF_ATTN, l, m, g);
        in.wait_bar = bar(b.qkv, l, 0);  // blocks 0..m of this layer
        in.wait_target = pp.n_qkv_n;
        in.wait_n = (uint16_t)(m + 1);
        in.wait_stride = 1;
        in.rel_bar = bar(b.attn, l, m);
        q.push_back(in);
      }
    end(s);
    s = begin();
    grouped(pp.n_o_n, [&](int m, uint32_t n) {
      Instr in = pf_make(PF_O, l, m, n);
      in.wait_bar = bar(b.attn, l, m);
      in.wait_target = (uint32_t)nkv;
      in.wait_n = 1;
      in.wait_stride = 1;
      in.rel_bar = bar(b.o, l, m);
      q.push_back(in);
    });
    end(s);
    s = begin();
    for (int m = 0; m < NB; ++m) {
      Instr in = pf_make(PF_NORM2, l, m, 0);
      in.wait_bar = bar(b.o, l, m);
      in.wait_target = pp.n_o_n;
      in.wait_n = 1;
      in.wait_stride = 1;
      in.rel_bar = bar(b.norm2, l, m);
      q.push_back(in);
    }
    end(s);
    s = begin();
    grouped(pp.n_gu_n, [&](int m, uint32_t n) {
      Instr in = pf_make(PF_GU, l, m, n);
      in.wait_bar = bar(b.norm2, l, m);
      in.wait_target = 1;
      in.wait_n = 1;
      in.wait_stride = 1;
      in.rel_bar = bar(b.gu, l, m);
      q.push_back(in);
    });
    end(s);
    s = begin();
    grouped(pp.n_down_n, [&](int m, uint32_t n) {
      Instr in = pf_make(PF_DOWN, l, m, n);
      in.wait_bar = bar(b.gu, l, m);
      in.wait_target = pp.n_gu_n;
      in.wait_n = 1;
      in.wait_stride = 1;
      in.rel_bar = bar(b.down, l, m);
      q.push_back(in);
    });
    end(s);
  }
  pp.n_body = (uint32_t)q.size();
  pp.n_perop_body = (uint32_t)pp.perop.size();
  // all-token logits: the final norm of every block, then the LM head (the
  // tensor-core GEMM of the normed rows with the [V][H] weights)
  uint32_t s = begin();
  for (int m = 0; m < NB; ++m) {
    Instr in = pf_make(PF_NORMF, L - 1, m, 0);
    in.wait_bar = bar(b.down, L - 1, m);
    in.wait_target = pp.n_down_n;
    in.wait_n = 1;
    in.wait_stride = 1;
    in.rel_bar = b.normf + (uint32_t)m;
    q.push_back(in);
  }
  end(s);
  s = begin();
  // (the normf and lm counters are released only by launches that run this
  // tail: they are cleared before each such launch and waited on absolutely)
  grouped(pp.n_lm_n, [&](int m, uint32_t n) {
    Instr in = pf_make(PF_LM, L - 1, m, n);
    in.flags = IF_ABS_TARGET;
    in.wait_bar = b.normf + (uint32_t)m;
    in.wait_target = 1;
    in.wait_n = 1;
    in.wait_stride = 1;
    in.rel_bar = b.lm + (uint32_t)m;
    q.push_back(in);
  });
  end(s);
  return MK_OK;
}

int simulate_prefill(const PrefillPlan& pp, const std::vector<Instr>& q, std::string* why) {
  std::vector<uint32_t> cnt(pp.bl.total, 0);
  for (size_t i = 0; i < q.size(); ++i) {
    const Instr& in = q[i];
    if (in.op < PF_NORM1 || in.op > PF_LM) {
      if (why) *why = "unknown prefill opcode at " + std::to_string(i);
      return MK_ERR_INVALID_ARG;
    }
    if (in.wait_bar != NO_BAR)
      for (uint32_t k = 0; k < in.wait_n; ++k) {
        const uint32_t b = in.wait_bar + k * in.wait_stride;
        if (b >= pp.bl.total || cnt[b] < in.wait_target) {
          if (why) *why = "prefill instruction " + std::to_string(i) + " waits before its producers";
          return MK_ERR_INVALID_ARG;
        }
      }
    if (in.rel_bar != NO_BAR) cnt[in.rel_bar] += 1;
  }
  for (size_t i = 0; i < q.size(); ++i) {
    const Instr& in = q[i];
    if (in.wait_bar == NO_BAR) continue;
    for (uint32_t k = 0; k < in.wait_n; ++k)
      if (cnt[in.wait_bar + k * in.wait_stride] != in.wait_target) {
        if (why) *why = "prefill barrier count mismatch at instruction " + std::to_string(i);
        return MK_ERR_INVALID_ARG;
      }
  }
  return MK_OK;
}

}  // namespace mk
