"""LM head and per-row statistics (fp64).

[MTP] section "Medusa：本体に複数の予測ヘッドを足す": the final hidden state h_t goes through one
LM head (a linear layer plus softmax) to give the distribution of the next token; [GLOSS]
architecture table: the original LM head has hidden_dim x vocab_size parameters.  The tree
forward therefore gives, at every node, z = W h (no bias) and p = softmax(z / tau).

Statistics of one row at temperature tau > 0 (y = z / tau):
    max   = max_v y_v,        LSE = log sum_v exp(y_v),
    p_v   = exp(y_v - LSE),   H   = -sum_v p_v ln p_v   (nats),
    argmax of z (lowest index on ties), and the gap between the two largest z values.
At tau = 0 (greedy) only the argmax and the gap are used; y = z is taken for the rest.
"""

import numpy as np


def logits(hidden_rows, W, chunk=4096):
    """z = W h for each row of ``hidden_rows`` [r][Hd]; W [V][Hd] (float32 or float64).

    W is widened to float64 one vocabulary chunk at a time; returns [r][V] float64.
    """
    H = np.asarray(hidden_rows, dtype=np.float64)
    V = W.shape[0]
    z = np.empty((H.shape[0], V))
    for v0 in range(0, V, chunk):
        z[:, v0: v0 + chunk] = H @ np.asarray(W[v0: v0 + chunk], dtype=np.float64).T
    return z


def softmax(y):
    m = y.max()
    e = np.exp(y - m)
    return e / e.sum()


def row_stats(z, tau):
    """Statistics of one logit row z [V] (float64).  Returns a dict."""
    z = np.asarray(z, dtype=np.float64)
    y = z / tau if tau > 0 else z.copy()
    m = y.max()
    lse = m + np.log(np.exp(y - m).sum())
    p = np.exp(y - lse)
    nz = p > 0
    H = -np.sum(p[nz] * np.log(p[nz]))
    am = int(np.argmax(z))  # first occurrence = lowest index
    rest = np.delete(z, am)
    gap = z[am] - rest.max() if rest.size else np.inf
    return dict(max=m, lse=lse, entropy=H, argmax=am, gap=gap, p=p)
