"""Pure-Python loop twin of the oracle, for tiny shapes only (test helper).

Every quantity is an explicit sum over scalar Python floats with math.exp;
it shares no code with oracle/evo_oracle.py.  Definition: the web page
"DeepSpeed4Science 技术指南 … Evoformer 内存高效注意力内核实战" §3.5 (scale,
add bias, softmax, times V) and §3.6-3.7 (bias shapes and both gradients).
"""
import math


def _bias(b1, b2, b, n, h, i, j):
    t = 0.0
    if b1 is not None:
        t += float(b1[b][n][0][0][j])
    if b2 is not None:
        t += float(b2[b][0][h][i][j])
    return t


def brute(q, k, v, b1, b2, do):
    """q, k, v, do: nested lists/arrays [B][N][L][H][D]; returns dict of nested lists."""
    B, N, L, H, D = len(q), len(q[0]), len(q[0][0]), len(q[0][0][0]), len(q[0][0][0][0])
    s = D ** -0.5
    z5 = lambda: [[[[[0.0] * D for _ in range(H)] for _ in range(L)] for _ in range(N)] for _ in range(B)]
    O, dQ, dK, dV = z5(), z5(), z5(), z5()
    LSE = [[[[0.0] * L for _ in range(H)] for _ in range(N)] for _ in range(B)]
    dB1 = [[[[[0.0] * L]] for _ in range(N)] for _ in range(B)]
    dB2 = [[[[[0.0] * L for _ in range(L)] for _ in range(H)]] for _ in range(B)]
    for b in range(B):
        for n in range(N):
            for h in range(H):
                x = [[s * sum(float(q[b][n][i][h][d]) * float(k[b][n][j][h][d]) for d in range(D))
                      + _bias(b1, b2, b, n, h, i, j) for j in range(L)] for i in range(L)]
                P = []
                for i in range(L):
                    mx = max(x[i])
                    if mx == -math.inf:
                        P.append([0.0] * L)
                        LSE[b][n][h][i] = -math.inf
                        continue
                    den = sum(math.exp(x[i][j] - mx) for j in range(L))
                    LSE[b][n][h][i] = mx + math.log(den)
                    P.append([math.exp(x[i][j] - mx) / den for j in range(L)])
                for i in range(L):
                    for d in range(D):
                        O[b][n][i][h][d] = sum(P[i][j] * float(v[b][n][j][h][d]) for j in range(L))
                for i in range(L):
                    delta = sum(float(do[b][n][i][h][d]) * O[b][n][i][h][d] for d in range(D))
                    for j in range(L):
                        dp = sum(float(do[b][n][i][h][d]) * float(v[b][n][j][h][d]) for d in range(D))
                        ds = P[i][j] * (dp - delta)
                        dB1[b][n][0][0][j] += ds
                        dB2[b][0][h][i][j] += ds
                        for d in range(D):
                            dQ[b][n][i][h][d] += s * ds * float(k[b][n][j][h][d])
                            dK[b][n][j][h][d] += s * ds * float(q[b][n][i][h][d])
                            dV[b][n][j][h][d] += P[i][j] * float(do[b][n][i][h][d])
    return {"o": O, "lse": LSE, "dq": dQ, "dk": dK, "dv": dV, "dbias1": dB1, "dbias2": dB2}
