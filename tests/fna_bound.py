"""Error bound for the FlashNormAttention forward's two bf16 tensor-core
operands, added to the elementwise tolerance of the parity tests.

The blog's §4 pseudocode (and the oracle) keeps ln_q and p = act(ln_q K^T)
unrounded.  The kernel feeds both matmuls bf16 operands, bf16(ln_q) and
bf16(act(s)), accumulates in fp32 and evaluates the activation with the
hardware tanh.  Per query row and head, to first order:

  ds_j = sum_d e_d k_jd               e_d:  rounding of ln_d,     |e_d| <= u |ln_d|
  dp_j = act'(s_j) ds_j + f_j + g_j   f_j:  rounding of act(s_j), |f_j| <= u |p_j|
                                      g_j:  tanh.approx error,    |g_j| <= t_j
  do_k = sum_j dp_j v_jk
       = sum_d e_d c_dk + sum_j f_j v_jk + sum_j g_j v_jk,   c_dk = sum_j act'(s_j) k_jd v_jk

(u = 2^-8 bounds the relative error of a round-to-nearest bf16 value.)  The
worst case, every term of both 128-long sums with the same sign, is about a
hundred times the error seen and larger than the outputs themselves, so it
checks nothing.  The bound used is the probabilistic one of Higham and Mary
("A New Approach to Probabilistic Rounding Error Analysis", SIAM J. Sci.
Comput. 41(5), 2019): the rounding errors e_d, f_j are modelled as
independent with mean zero, and Hoeffding's inequality bounds their weighted
sum by lambda sigma_k,

  sigma_k^2 = sum_d (u ln_d c_dk)^2 + sum_j (u p_j v_jk)^2,

except with probability 2 exp(-lambda^2 / 2) (lambda = 8: 2.5e-14 per
element).  The tanh error g_j (both activations are written h + h tanh(.),
h = s / 2; tanh.approx is within about 2^-11, taken as 2^-10) and fp32
accumulation (2^-17 of the absolute sums, 128 terms) are not modelled as
random: they enter with their worst case.  With E_k = lambda sigma_k + the two
worst-case terms, the RMSNorm over all heads (y = o r, r = (mean(o^2) +
eps2)^-1/2) gives dy_k = r (do_k - y_k mean(y do)).  mean(y do) is again a
weighted sum of the same rounding errors (weights (1/n) sum_k y_k c_dk and
(1/n) sum_k y_k v_jk), bounded the same way by lambda sigma_m, plus the
worst-case terms' rms.  So

  |dy_k| <= 1.1 r (E_k + |y_k| (lambda sigma_m + rms(T + A)))

(1.1 for second-order terms, which are about u times the first-order ones).
The test adds this to 2e-2 + 1.6e-2 |ref|; the residual q and the output's own
bf16 rounding are covered by that base bound.

Everything here is fp64 numpy on the test's inputs; nothing comes from the
CUDA path.
"""
import numpy as np

import nf_inputs

U_BF16 = 2.0 ** -8
ACC = 2.0 ** -17
TANH_ERR = 2.0 ** -10
LAMBDA = 8.0
GELU_C = np.sqrt(2.0 / np.pi)


def _act(s, act):
    if act == 1:
        return 0.5 * s * (1.0 + np.tanh(GELU_C * (s + 0.044715 * s ** 3)))
    if act == 2:
        return s / (1.0 + np.exp(-s))
    return s


def _act_slope(s, act):
    if act == 1:
        t = np.tanh(GELU_C * (s + 0.044715 * s ** 3))
        return 0.5 * (1.0 + t) + 0.5 * s * (1.0 - t * t) * GELU_C * (1.0 + 3 * 0.044715 * s * s)
    if act == 2:
        sg = 1.0 / (1.0 + np.exp(-s))
        return sg * (1.0 + s * (1.0 - sg))
    return np.ones_like(s)


def operand_bound(Q, K, V, act, eps1, eps2, q_len=None, chunk=128):
    """Per-element extra bound [B, Lq, H, D] (zero on rows past q_len)."""
    q = nf_inputs.bf16_to_f64(Q)
    k = nf_inputs.bf16_to_f64(K)
    v = nf_inputs.bf16_to_f64(V)
    B, Lq, H, D = q.shape
    n_all = H * D
    x = q.reshape(B, Lq, n_all)
    mu = x.mean(-1, keepdims=True)
    ln = ((x - mu) / np.sqrt(((x - mu) ** 2).mean(-1, keepdims=True) + eps1)).reshape(B, Lq, H, D)
    out = np.zeros((B, Lq, H, D))
    for b in range(B):
        n = Lq if q_len is None else int(q_len[b])
        for r0 in range(0, n, chunk):
            r1 = min(n, r0 + chunk)
            R = r1 - r0
            lnc = ln[b, r0:r1]                                           # [R, H, D]
            s = np.einsum("rhd,jhd->rhj", lnc, k[b])                     # [R, H, Lkv]
            p = _act(s, act)
            O = np.einsum("rhj,jhd->rhd", p, v[b]) + lnc
            rr = 1.0 / np.sqrt((O * O).reshape(R, n_all).mean(-1) + eps2)  # [R]
            y = O * rr[:, None, None]
            sig2 = np.empty((R, H, D))
            wc = np.empty((R, H, D))                                     # tanh + accumulation, worst case
            sig2_m = np.zeros(R)
            for h in range(H):
                lnh, sh, ph, yh = lnc[:, h], s[:, h], p[:, h], y[:, h]
                kh, vh = k[b, :, h], v[b, :, h]                          # [Lkv, D]
                a = _act_slope(sh, act)
                c = np.matmul(kh.T[None] * a[:, None, :], vh[None])      # [R, D, D]: c_dk
                ul, up = U_BF16 * lnh, U_BF16 * ph
                sig2[:, h] = np.einsum("rd,rdk->rk", ul * ul, c * c) + (up * up) @ (vh * vh)
                cm_l = np.einsum("rdk,rk->rd", c, yh) / n_all            # weight of e_d in mean(y do)
                cm_p = (yh @ vh.T) / n_all                               # weight of f_j in mean(y do)
                sig2_m += ((ul * cm_l) ** 2).sum(-1) + ((up * cm_p) ** 2).sum(-1)
                va = np.abs(vh)
                t = (0.5 * np.abs(sh) * TANH_ERR) @ va if act != 0 else 0.0
                acc = (ACC * (np.abs(a) * (np.abs(lnh) @ np.abs(kh).T) + np.abs(ph))) @ va
                wc[:, h] = t + acc
            E = LAMBDA * np.sqrt(sig2) + wc
            m = LAMBDA * np.sqrt(sig2_m) + np.sqrt((wc * wc).reshape(R, n_all).mean(-1))
            out[b, r0:r1] = 1.1 * rr[:, None, None] * (E + np.abs(y) * m[:, None, None])
    return out
