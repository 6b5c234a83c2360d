"""Independent full-sequence references used to pin the CPU oracle.

The oracle decodes one token at a time with a KV cache.  These references
compute every position at once (prefill style) in float64 with library
routines: ``torch.nn.functional.scaled_dot_product_attention`` with an
explicit causal / sliding-window mask, ``torch.nn.functional.rms_norm``,
``torch.nn.functional.silu``, RoPE as a complex rotation (the pair (c, c+dh/2)
read as the complex number x_c + i x_{c+dh/2}), and FP16 rounding of K and V by
numpy's ``astype(float16)`` (a single correctly rounded step; torch's float64
to float16 cast rounds twice, through float32).  None of this code is shared with the
oracle or with the CUDA engine.
"""
from __future__ import annotations

import numpy as np
import torch
import torch.nn.functional as F

import synth


def _weights(shape, blob):
    return {k: torch.from_numpy(np.asarray(v, dtype=np.float64)) for k, v in
            synth.weight_views(shape, blob).items()}


def _rope_complex(x: torch.Tensor, pos: torch.Tensor, theta: float) -> torch.Tensor:
    """x [n, H, dh] rotated at positions pos [n] (rotate-half pairing)."""
    dh = x.shape[-1]
    half = dh // 2
    z = torch.complex(x[..., :half], x[..., half:])
    freq = theta ** (-2.0 * torch.arange(half, dtype=torch.float64) / dh)
    rot = torch.polar(torch.ones(len(pos), half, dtype=torch.float64),
                      pos.to(torch.float64)[:, None] * freq[None, :])
    z = z * rot[:, None, :]
    return torch.cat([z.real, z.imag], dim=-1)


def _mask(q_pos: torch.Tensor, k_pos: torch.Tensor, window: int) -> torch.Tensor:
    allowed = k_pos[None, :] <= q_pos[:, None]
    if window > 0:
        allowed &= k_pos[None, :] > (q_pos[:, None] - window)
    return allowed


def _attend(q, k, v, q_pos, k_pos, window):
    """q [n, Hq, dh]; k, v [m, Hq, dh] (already expanded per q head)."""
    mask = _mask(q_pos, k_pos, window)
    out = F.scaled_dot_product_attention(q.transpose(0, 1), k.transpose(0, 1), v.transpose(0, 1),
                                         attn_mask=mask[None])
    return out.transpose(0, 1)


class _Ctx:
    def __init__(self, shape, blob, tokens, round_kv, kv_prefix, n_prefix):
        self.m = shape
        self.W = _weights(shape, blob)
        self.round_kv = round_kv
        self.tok = torch.as_tensor(np.asarray(tokens, dtype=np.int64))
        self.n0 = n_prefix
        self.pos = torch.arange(n_prefix, n_prefix + len(tokens))
        self.k_pos = torch.arange(0, n_prefix + len(tokens))
        self.prefix = None
        if kv_prefix is not None and n_prefix > 0:
            m = shape
            kv = np.asarray(kv_prefix, dtype=np.uint16).view(np.float16).astype(np.float64)
            self.prefix = torch.from_numpy(kv.reshape(m.n_layers, 2, n_prefix, m.n_kv_heads, m.head_dim))

    def rnd(self, t):
        if not self.round_kv:
            return t
        return torch.from_numpy(t.numpy().astype(np.float16).astype(np.float64))

    def attention(self, l, h, q_heads):
        """Attention of layer l for the given q heads, from normed input h [n, d].
        Returns the concatenated head outputs [n, len(q_heads)*dh]."""
        m, W = self.m, self.W
        dh, group = m.head_dim, m.n_q_heads // m.n_kv_heads
        Wq, Wk, Wv = (W[f"{n}.{l}"].reshape(-1, dh, m.d_model) for n in ("Wq", "Wk", "Wv"))
        kv_heads = sorted({hq // group for hq in q_heads})
        q = torch.einsum("hcd,nd->nhc", Wq[q_heads], h)
        k = torch.einsum("hcd,nd->nhc", Wk[kv_heads], h)
        v = torch.einsum("hcd,nd->nhc", Wv[kv_heads], h)
        q = _rope_complex(q, self.pos, m.rope_theta)
        k = self.rnd(_rope_complex(k, self.pos, m.rope_theta))
        v = self.rnd(v)
        if self.prefix is not None:
            k = torch.cat([self.prefix[l, 0][:, kv_heads], k], dim=0)
            v = torch.cat([self.prefix[l, 1][:, kv_heads], v], dim=0)
        sel = [kv_heads.index(hq // group) for hq in q_heads]
        o = _attend(q, k[:, sel], v[:, sel], self.pos, self.k_pos, m.swa_window[l])
        return o.reshape(len(self.pos), -1)

    def ffn(self, l, h, units):
        W = self.W
        a = h @ W[f"Wg.{l}"][units].T
        b = h @ W[f"Wu.{l}"][units].T
        return F.silu(a) * b

    def norm(self, x, g):
        return F.rms_norm(x, (self.m.d_model,), weight=g, eps=self.m.rms_eps)


def standard_transformer(shape, blob, tokens, round_kv=True, kv_prefix=None, n_prefix=0):
    """Textbook pre-norm GQA decoder with per-layer residual adds (no lanes, no
    delay).  Returns logits [n, vocab] for every position of ``tokens``."""
    c = _Ctx(shape, blob, tokens, round_kv, kv_prefix, n_prefix)
    m, W = c.m, c.W
    x = W["E"][c.tok]
    all_q = list(range(m.n_q_heads))
    for l in range(m.n_layers):
        x = x + c.attention(l, c.norm(x, W[f"g_attn.{l}"]), all_q) @ W[f"Wo.{l}"].T
        x = x + c.ffn(l, c.norm(x, W[f"g_ffn.{l}"]), torch.arange(m.ffn_dim)) @ W[f"Wd.{l}"].T
    return (c.norm(x, W["g_f"]) @ W["W_lm"].T).numpy()


def closed_form_all_read_embedding(shape, blob, tokens, round_kv=True):
    """Logits when every sub-block reads the embedding alone, which the
    delayed lane sum gives when 2*delay + 1 >= 2*n_layers:
        logits = W_lm rmsnorm(e + sum_l [attn_l(norm e) + ffn_l(norm e)])."""
    c = _Ctx(shape, blob, tokens, round_kv, None, 0)
    m, W = c.m, c.W
    e = W["E"][c.tok]
    out = e.clone()
    for l in range(m.n_layers):
        out = out + c.attention(l, c.norm(e, W[f"g_attn.{l}"]), list(range(m.n_q_heads))) @ W[f"Wo.{l}"].T
        out = out + c.ffn(l, c.norm(e, W[f"g_ffn.{l}"]), torch.arange(m.ffn_dim)) @ W[f"Wd.{l}"].T
    return (c.norm(out, W["g_f"]) @ W["W_lm"].T).numpy()


def delayed_lanes(shape, blob, tokens, round_kv=True):
    """Prefill-style evaluation of the delayed lane sum with explicit lanes.

    Sub-block s reads x(s) = e + sum over u <= s-1-2d of every lane's partial
    (plus, with own_lane_immediate, the lane's own partials for u <= s-1).
    Computed for all positions at once, lane by lane."""
    c = _Ctx(shape, blob, tokens, round_kv, None, 0)
    m, W = c.m, c.W
    NL, d, dh = m.n_lanes, m.dtp_delay, m.head_dim
    hq, fl = m.n_q_heads // NL, m.ffn_dim // NL
    e = W["E"][c.tok]
    parts = []  # parts[u][i] -> [n, d_model]
    for s in range(2 * m.n_layers):
        l = s // 2
        row = []
        for i in range(NL):
            x = e.clone()
            for u in range(s):
                for j in range(NL):
                    if u <= s - 1 - 2 * d or (m.own_lane_immediate and j == i):
                        x = x + parts[u][j]
            if s % 2 == 0:
                heads = list(range(i * hq, (i + 1) * hq))
                o = c.attention(l, c.norm(x, W[f"g_attn.{l}"]), heads)
                row.append(o @ W[f"Wo.{l}"][:, i * hq * dh:(i + 1) * hq * dh].T)
            else:
                units = torch.arange(i * fl, (i + 1) * fl)
                u_ = c.ffn(l, c.norm(x, W[f"g_ffn.{l}"]), units)
                row.append(u_ @ W[f"Wd.{l}"][:, i * fl:(i + 1) * fl].T)
        parts.append(row)
    x = e + sum(p for row in parts for p in row)
    return (c.norm(x, W["g_f"]) @ W["W_lm"].T).numpy()
