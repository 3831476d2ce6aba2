"""Worker of the full-output oracle checks: one (batch, query head) of the
float64 causal attention oracle per task, in a spawned process that imports
numpy and the oracle only (one BLAS thread per process, set before numpy
loads)."""
import os

for _var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ[_var] = "1"

import numpy as np  # noqa: E402

from oracle import attention as oattn  # noqa: E402


def head_output(task):
    """task = (q [S,Dqk], k [S,Dqk], v [S,Dv], scale) -> O [S,Dv] float64."""
    q, k, v, scale = task
    return oattn.causal_attention(q[None, :, None], k[None, :, None], v[None, :, None], scale)[0, :, 0]
