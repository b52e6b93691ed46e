"""Helpers shared by the GPU parity tests (not a test module)."""
import math

import numpy as np
import torch

import attn_inputs as gen
from oracle import attn64

O_TOL = 1e-2      # max |O_gpu - O_oracle|
LSE_TOL = 1e-3    # max |LSE_gpu - LSE_oracle|
GRAD_TOL = 2e-2   # ||G_gpu - G_oracle||_F / ||G_oracle||_F for dQ, dK, dV


# Largest error seen per (workload, quantity), written out at the end of the
# session when ATTN_PARITY_REPORT names a file (tests/conftest.py).
REPORT = {}


def record(workload, key, value):
    cur = REPORT.setdefault(workload, {})
    cur[key] = max(cur.get(key, 0.0), float(value))


def lib():
    import exact_attention_66_gb300 as ea
    return ea


def inputs(B, Hq, Hkv, N, d, seed, doc=False):
    x = gen.make_inputs(B, Hq, Hkv, N, d, seed, doc=doc)
    if doc:
        x["doc_ids_np"] = x["doc_ids"]
    return x


def mods_pair(x, causal=False, window=None, doc=False, softcap=None, alibi=False):
    """(library mods, oracle mods) for the same mask/score mods."""
    ea = lib()
    dev_doc = torch.from_numpy(x["doc_ids_np"]).cuda() if doc else None
    m = ea.make_mods(causal=causal, window=window, doc_ids=dev_doc, softcap=softcap, alibi=alibi)
    om = attn64.Mods(causal=causal, window=window, doc_ids=x["doc_ids_np"] if doc else None,
                     softcap=softcap, alibi=alibi)
    return m, om


def to_dev(x):
    return {k: v.cuda() for k, v in x.items() if isinstance(v, torch.Tensor)}


def max_abs(a, b):
    return float(np.abs(np.asarray(a, np.float64) - np.asarray(b, np.float64)).max())


def rel_fro(a, b):
    """||a - b||_F / ||b||_F, the denominator floored at an RMS of 1e-3 (for an
    all-but-zero truth, e.g. dQ with a single key, the error is then absolute)."""
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-3 * np.sqrt(b.size)))


def default_scale(d):
    return 1.0 / math.sqrt(d)
