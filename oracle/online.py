"""The tiled online-softmax recurrence and the split merge, in float64.

Second, independent oracle path, used only to pin ``oracle.attention`` and to
state the merge the GPU split-K path relies on (test infrastructure only).

Recurrence [Ch15 §15.1 算法详解; Deploy §4.1 FlashAttention (m(x), l(x))]:
for one query block and key/value tiles j = 1..Tc,
    S_j      = Q K_j^T / sqrt(d)
    m^(j)    = max(m^(j-1), rowmax(S_j))
    alpha^(j)= exp(m^(j-1) - m^(j))
    P_j      = exp(S_j - m^(j))
    l^(j)    = alpha^(j) l^(j-1) + rowsum(P_j)
    O^(j)    = diag(alpha^(j)) O^(j-1) + P_j V_j
starting from m = -inf, l = 0, O = 0, and O = diag(l)^-1 O at the end.

Split merge (split-K over the context) [Deploy §2.5 LMDeploy, "2. TurboMind 推理引擎解析"
names Split-K decoding but does not spell out the combination; it is the
same alpha rescaling applied once to whole partial states]: partial states
(m_k, l_k, O_k) over disjoint key ranges combine as
    M = max_k m_k,  L = sum_k l_k exp(m_k - M),  O = sum_k O_k exp(m_k - M) / L.
"""

import numpy as np


def partial_state(q, k, v, scale, tile):
    """Run the recurrence over all of k/v in tiles of ``tile`` keys.

    q [nq, D]; k, v [n, D] (float64).  Returns the unnormalised state (m, l, O)
    with m, l of shape [nq] and O of shape [nq, D].
    """
    nq, d = q.shape
    dt = q.dtype  # float64 normally; float32 only to rerun the pages' fp32 check
    m = np.full(nq, -np.inf, dtype=dt)
    l = np.zeros(nq, dtype=dt)
    o = np.zeros((nq, d), dtype=dt)
    for j0 in range(0, k.shape[0], tile):
        kj = k[j0:j0 + tile]
        vj = v[j0:j0 + tile]
        s = (q @ kj.T) * dt.type(scale)
        m_new = np.maximum(m, s.max(axis=1))
        alpha = np.exp(m - m_new)
        p = np.exp(s - m_new[:, None])
        l = alpha * l + p.sum(axis=1)
        o = alpha[:, None] * o + p @ vj
        m = m_new
    return m, l, o


def finish(state):
    m, l, o = state
    return o / l[:, None]


def merge(states):
    """Combine partial states over disjoint key ranges into the final output."""
    ms = np.stack([s[0] for s in states])      # [K, nq]
    big_m = ms.max(axis=0)
    w = np.exp(ms - big_m[None, :])
    big_l = sum(w[i] * states[i][1] for i in range(len(states)))
    o = sum(w[i][:, None] * states[i][2] for i in range(len(states)))
    return o / big_l[:, None]


def attention_online(q, k, v, scale, tile):
    return finish(partial_state(q, k, v, scale, tile))


def attention_split(q, k, v, scale, tile, split):
    """Split the keys into ranges of ``split`` keys, run the recurrence on each, merge."""
    states = [partial_state(q, k[a:a + split], v[a:a + split], scale, tile)
              for a in range(0, k.shape[0], split)]
    return merge(states)
