"""A small exactly-specified problem whose inputs are bf16-exact rationals (no RNG, so it is
the same on every platform). ``python tests/golden/rational_case.py`` rewrites
``rational_case.json`` from the fp64 oracle alone; tests compare the oracle and the CUDA
library against it.

The pages print no worked example of the loss, so this fixture is an oracle-written
regression value, not a published one.
"""
import json
import os
import sys

import numpy as np

N, D_S, D_T, V, TAU, GRAD_SCALE = 5, 16, 24, 40, 1.25, 1.0


def inputs():
    n = np.arange(N)[:, None]
    v = np.arange(V)[:, None]
    js = np.arange(D_S)[None, :]
    jt = np.arange(D_T)[None, :]
    h_s = ((3 * n + 5 * js) % 17 - 8) / 8.0
    W_s = ((7 * v + 2 * js) % 13 - 6) / 32.0
    h_t = ((5 * n + 3 * jt) % 19 - 9) / 8.0
    W_t = ((11 * v + jt) % 23 - 11) / 64.0
    return h_s, W_s, h_t, W_t


def main():
    here = os.path.dirname(os.path.abspath(__file__))
    sys.path.insert(0, os.path.dirname(os.path.dirname(here)))
    from oracle import kl_oracle as orc
    h_s, W_s, h_t, W_t = inputs()
    kl, lse_s, lse_t, loss = orc.kl_forward(h_s, W_s, h_t, W_t, TAU)
    dh, dW = orc.kl_backward(h_s, W_s, h_t, W_t, TAU, grad_scale=GRAD_SCALE)
    out = {"N": N, "d_s": D_S, "d_t": D_T, "V": V, "tau": TAU, "grad_scale": GRAD_SCALE,
           "kl": kl.tolist(), "lse_s": lse_s.tolist(), "lse_t": lse_t.tolist(), "loss": loss,
           "dh_s": dh.tolist(), "dW_s": dW.tolist()}
    with open(os.path.join(here, "rational_case.json"), "w") as f:
        json.dump(out, f, indent=0)


if __name__ == "__main__":
    main()
