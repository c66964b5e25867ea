"""Parity at large sizes: the WS matvecs with 2,097,152 rows (16384 row blocks, so the grid
runs in many waves) and M = 16, a ragged row count beyond it, and a probe far wider than the
7424-wide workload."""
import ctypes

import numpy as np
import pytest
import torch

from dspark_draft_sampling_gb300 import api, synth
from tests import parity

pytestmark = pytest.mark.gpu

MAX_N = 16384 * 128  # 16384 row blocks of 128 rows


@pytest.fixture(scope="module", autouse=True)
def _lib(dspark_lib):
    return dspark_lib


def test_fp16_matvec_at_max_rows_and_m():
    inp = synth.ws_inputs(16, MAX_N, 8, seed=1, w_sd=0.5)
    W = torch.from_numpy(inp["W"].view(np.int16)).cuda().view(torch.float16)
    X = torch.from_numpy(inp["X"].view(np.int16)).cuda().view(torch.float16)
    y = api.ws_matvec(W, X, out_fp32=True)
    torch.cuda.synchronize()
    parity.check_ws(inp, y32=y.cpu().numpy())


def test_fp16_matvec_ragged_rows_beyond_max_sampled():
    """One row block and one row more (a partial last block): a seeded sample of 4096 weight
    rows, plus the last 129, against the oracle (each output row depends only on its own
    weights)."""
    N, K, M = MAX_N + 129, 64, 16
    inp = synth.ws_inputs(M, N, K, seed=2, w_sd=0.5)
    W = torch.from_numpy(inp["W"].view(np.int16)).cuda().view(torch.float16)
    X = torch.from_numpy(inp["X"].view(np.int16)).cuda().view(torch.float16)
    y = api.ws_matvec(W, X, out_fp32=True)
    torch.cuda.synchronize()
    rows = np.unique(np.concatenate([np.random.default_rng(3).choice(N, 4096, replace=False),
                                     np.arange(N - 129, N)]))
    sub = dict(W=np.ascontiguousarray(inp["W"][rows]), X=inp["X"], M=M, N=len(rows), K=K)
    parity.check_ws(sub, y32=y.cpu().numpy()[:, rows])


def test_q8_matvec_at_max_rows_and_m_sampled():
    """2,097,152 x 256 Q8_0 weights (544 MB) against 16 rows of X; the oracle checks a
    seeded sample of 4096 weight rows (every output row depends only on its own weights)."""
    N, K, M = MAX_N, 256, 16
    inp = synth.ws_q8_inputs(M, N, K, seed=2)
    q, d = api.q8_0_repack(torch.from_numpy(inp["Wq8"]).cuda(), N, K)
    X = torch.from_numpy(inp["X"].view(np.int16)).cuda().view(torch.float16)
    y = api.ws_matvec_q8(q, d, X, out_fp32=True)
    torch.cuda.synchronize()
    rows = np.sort(np.random.default_rng(3).choice(N, 4096, replace=False))
    blocks = inp["Wq8"].reshape(N, K // 32 * 34)[rows].reshape(-1)
    sub = dict(Wq8=blocks, X=inp["X"], M=M, N=len(rows), K=K)
    parity.check_ws_q8(sub, y32=y.cpu().numpy()[:, rows])


def test_probe_far_wider_than_the_workload():
    inp = synth.probe_inputs(5, 32768 * 4, seed=4, random_scales=True, scale=0.002)
    z, gate = parity.gpu_probe(inp)
    parity.check_probe(inp, z, gate)
