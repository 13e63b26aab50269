"""Pure-Python loop forward of the bidirectional transformer, for tiny sizes.

Written from the textbook definitions with plain lists and the math module
(no numpy), independently of the oracle, to pin the oracle's vectorised
forward: a dropped term, a wrong sign, a swapped index or a transposed
operand in either shows up as a mismatch.  Used by the oracle pin tests only.
"""
import math
import struct


def bf16(x):
    """Nearest bfloat16 (ties to even) of a Python float, via its float32 bits."""
    (u,) = struct.unpack("<I", struct.pack("<f", x))
    lsb = (u >> 16) & 1
    u = (u + 0x7FFF + lsb) & 0xFFFF0000
    (f,) = struct.unpack("<f", struct.pack("<I", u & 0xFFFFFFFF))
    return f


def _mat(w):
    return [[float(v) for v in row] for row in w]


def matvec(W, x):
    # W [out][in], x [in] -> [out]
    return [sum(W[o][i] * x[i] for i in range(len(x))) for o in range(len(W))]


def rms(x, g, eps):
    s = math.sqrt(sum(v * v for v in x) / len(x) + eps)
    return [x[i] / s * g[i] for i in range(len(x))]


def rot(vec, p, theta):
    hd = len(vec)
    half = hd // 2
    out = [0.0] * hd
    for i in range(half):
        a = p * theta ** (-2.0 * i / hd)
        out[i] = vec[i] * math.cos(a) - vec[i + half] * math.sin(a)
        out[i + half] = vec[i + half] * math.cos(a) + vec[i] * math.sin(a)
    return out


def silu(v):
    return v / (1.0 + math.exp(-v))


def swiglu(wg, wu, wd, a, R):
    """(silu(a Wg^T) * a Wu^T) Wd^T with the product rounded by R."""
    gg, uu = matvec(wg, a), matvec(wu, a)
    act = [R(silu(gg[i]) * uu[i]) for i in range(len(gg))]
    return matvec(wd, act)


def moe(desc, router, w13, w2, a, R):
    """Mixture of experts for one row: softmax over all experts' router
    logits; the top_k experts by probability (lower index first on equal
    probability) each add p_e times their own SwiGLU output; the selected
    probabilities are used as they are (no renormalisation)."""
    E, k, fe = desc.n_experts, desc.top_k, desc.expert_ffn
    logit = matvec(router, a)
    top = max(logit)
    ex = [math.exp(v - top) for v in logit]
    z = sum(ex)
    p = [v / z for v in ex]
    order = sorted(range(E), key=lambda e: (-p[e], e))
    out = [0.0] * len(a)
    for e in order[:k]:
        y = swiglu(w13[e][:fe], w13[e][fe:], w2[e], a, R)
        for i in range(len(a)):
            out[i] += p[e] * y[i]
    return out


def forward_logits(desc, weights, ids, bf16_mode=False):
    """Full forward of one sequence ids [L]; returns logits [L][V] (mask logit -inf).

    weights: list in pointer order (dense or mixture-of-experts layers), as
    nested lists.
    """
    R = bf16 if bf16_mode else (lambda v: v)
    d, H, hd = desc.d_model, desc.n_heads, desc.head_dim
    L = len(ids)
    E = _mat(weights[0])
    h = [list(E[t]) for t in ids]
    for l in range(desc.n_layers):
        b = 1 + 9 * l
        g1, wq, wk, wv, wo, g2, wg, wu, wd = weights[b:b + 9]
        g1, g2 = [float(v) for v in g1], [float(v) for v in g2]
        wq, wk, wv, wo = map(_mat, (wq, wk, wv, wo))
        if getattr(desc, "n_experts", 0):   # router [E][d], w13 [E][2fe][d], w2 [E][d][fe]
            wg, wu, wd = _mat(wg), [_mat(m) for m in wu], [_mat(m) for m in wd]
        else:
            wg, wu, wd = map(_mat, (wg, wu, wd))
        Q, K, V = [], [], []
        for t in range(L):
            a = [R(v) for v in rms(h[t], g1, desc.rms_eps)]
            q, k, v = matvec(wq, a), matvec(wk, a), matvec(wv, a)
            qh, kh = [], []
            for j in range(H):
                qh += rot(q[j * hd:(j + 1) * hd], t, desc.rope_theta)
                kh += rot(k[j * hd:(j + 1) * hd], t, desc.rope_theta)
            Q.append([R(x) for x in qh])
            K.append([R(x) for x in kh])
            V.append([R(x) for x in v])
        newh = []
        for t in range(L):
            o = [0.0] * d
            for j in range(H):
                sl = slice(j * hd, (j + 1) * hd)
                sc = [sum(x * y for x, y in zip(Q[t][sl], K[u][sl])) / math.sqrt(hd) for u in range(L)]
                m = max(sc)
                ex = [math.exp(s - m) for s in sc]
                z = sum(ex)
                for c in range(hd):
                    o[j * hd + c] = sum(ex[u] / z * V[u][j * hd + c] for u in range(L))
            o = [R(x) for x in o]
            ho = matvec(wo, o)
            ht = [h[t][i] + ho[i] for i in range(d)]
            a = [R(v) for v in rms(ht, g2, desc.rms_eps)]
            if getattr(desc, "n_experts", 0):
                dn = moe(desc, wg, wu, wd, a, R)
            else:
                dn = swiglu(wg, wu, wd, a, R)
            newh.append([ht[i] + dn[i] for i in range(d)])
        h = newh
    gf = [float(v) for v in weights[1 + 9 * desc.n_layers]]
    lm = _mat(weights[2 + 9 * desc.n_layers])
    out = []
    for t in range(L):
        a = [R(v) for v in rms(h[t], gf, desc.rms_eps)]
        lg = [desc.logit_scale * x for x in matvec(lm, a)]
        lg[desc.mask_id] = -math.inf
        out.append(lg)
    return out
