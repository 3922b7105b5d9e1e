"""The bench's MoE and dense steps as they are timed: weight quantizations run on a side stream
joined by events, and the output must be bit-identical to the same launches run in order on one
stream (the GEMMs accumulate in a fixed order, so any missing join would show)."""
import importlib.util
import os

import pytest
import torch

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("nvq_bench", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_moe_step_concurrent_equals_serial():
    import nvfp4_quantization_block_gb300 as nvq
    import workloads
    b = _bench()
    dev = torch.device("cuda:0")
    W = b.WORKLOADS["moe"](torch, nvq, workloads, dev)
    x, w1, w2 = W["inputs"]
    poison = (w1 * 3.0, w2 * 0.25)            # other weights: every intermediate buffer changes
    timer = b.Timer(torch)
    outs = []
    for active in (False, True, False):
        timer.active = True                   # the poisoning step in order on one stream
        W["step"](timer, [x], poison)
        torch.cuda.synchronize()
        timer.active = active                 # inactive: the timed schedule (side stream + joins)
        res = W["step"](timer, [x], (w1, w2))
        torch.cuda.synchronize()
        outs.append([o.clone() for o in res])
    for other in outs[1:]:
        for u, v in zip(outs[0], other):
            assert torch.equal(u.view(torch.int16), v.view(torch.int16))


def test_dense_step_concurrent_equals_serial():
    import nvfp4_quantization_block_gb300 as nvq
    import workloads
    b = _bench()
    dev = torch.device("cuda:0")
    W = b.WORKLOADS["dense"](torch, nvq, workloads, dev)
    x, w = W["inputs"]
    timer = b.Timer(torch)
    outs = []
    for active in (False, True, False):
        timer.active = True
        W["step"](timer, x * 0.5, w * 2.0)    # other inputs: every intermediate buffer changes
        torch.cuda.synchronize()
        timer.active = active
        res = W["step"](timer, x, w)
        torch.cuda.synchronize()
        outs.append([o.clone() for o in res])
    for other in outs[1:]:
        for u, v in zip(outs[0], other):
            assert torch.equal(u.view(torch.int16), v.view(torch.int16))
