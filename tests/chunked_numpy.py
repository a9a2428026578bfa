"""The chunked (parallel-in-chunk, sequential-across-chunks) form of the
Mamba-3 recurrence, written in plain fp64 numpy for the tests.

It restates the decomposition the CUDA path uses, so that the tests can check
that decomposition against the sequential oracle on tiny inputs (any chunk
length, ragged last chunk, nonzero initial state and carry):

* inside a chunk, everything is expressed in a frame rotated by the
  chunk-local cumulative angle phi_t = sum_{s0<=u<=t} dt_u theta_u, so the
  complex transition becomes a real scalar decay and the rotation moves onto
  B and C (data-dependent RoPE; linkstar.cloud/article/869, section
  "RoPE技巧");
* the in-chunk operator is the product of a 1-semiseparable decay matrix and
  the 2-band trapezoid matrix (same page, section "第一刀", "它可以用并行形式
  计算"), so token j < t contributes with weight
  exp(cA_t - cA_j) * (lambda_j dt_j + (1 - lambda_{j+1}) dt_{j+1}) and token t
  itself with lambda_t dt_t;
* between chunks the N x P state is carried in fp64 and rotated back to the
  true frame by the chunk's total angle (chunked algorithm; linkstar.cloud
  article, section "训练怎么办").
"""
import numpy as np


def rot(v, c, s):
    """Rotate adjacent pairs (v[..., 2k], v[..., 2k+1]) by the angle with cosine c, sine s.

    c, s broadcast against v[..., ::2].  R(phi) = [[cos, -sin], [sin, cos]].
    """
    out = np.empty_like(v)
    a, b = v[..., 0::2], v[..., 1::2]
    out[..., 0::2] = c * a - s * b
    out[..., 1::2] = s * a + c * b
    return out


def scan_chunked(x, B, C, dt, A, lam, theta, h0=None, Bprev=None, xprev=None, Q=64):
    bsz, L, H, R, P = x.shape
    N = B.shape[-1]
    y = np.zeros((bsz, L, H, R, P))
    h_out = np.zeros((bsz, H, N, P))
    for b in range(bsz):
        for h in range(H):
            d, a_, l_ = dt[b, :, h], A[b, :, h], lam[b, :, h]
            g = l_ * d
            w = g.copy()
            w[:-1] += (1.0 - l_[1:]) * d[1:]
            S = np.zeros((N, P)) if h0 is None else h0[b, h].copy()
            if Bprev is not None and L > 0:
                S = S + (1.0 - l_[0]) * d[0] * (Bprev[b, h].T @ xprev[b, h])
            for s0 in range(0, L, Q):
                e = min(s0 + Q, L)
                ca = np.cumsum(d[s0:e] * a_[s0:e])                         # [Qc]
                phi = np.cumsum(d[s0:e, None] * theta[b, s0:e, h], axis=0)  # [Qc, N/2]
                c, s = np.cos(phi), np.sin(phi)
                Bb = rot(B[b, s0:e, h], c[:, None, :], -s[:, None, :])      # R(-phi) B
                Cb = rot(C[b, s0:e, h], c[:, None, :], -s[:, None, :])
                X = x[b, s0:e, h]                                           # [Qc, R, P]
                Qc = e - s0
                M = np.zeros((Qc, Qc))
                for t in range(Qc):
                    for j in range(t):
                        M[t, j] = np.exp(ca[t] - ca[j]) * w[s0 + j]
                    M[t, t] = g[s0 + t]
                G = np.einsum("trn,jqn->trjq", Cb, Bb) * M[:, None, :, None]
                y[b, s0:e, h] = np.einsum("trjq,jqp->trp", G, X) + \
                    np.exp(ca)[:, None, None] * np.einsum("trn,np->trp", Cb, S)
                wt = np.exp(ca[-1] - ca) * w[s0:e]
                S = np.exp(ca[-1]) * S + np.einsum("j,jqn,jqp->np", wt, Bb, X)
                S = rot(S.T, c[-1], s[-1]).T                                # back to the true frame
            h_out[b, h] = S
    return y, h_out
