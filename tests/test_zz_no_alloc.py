"""kda_chunk_forward_split_noalloc: the split chunked forward for callers that cannot allocate
device memory during the call (a serving runtime that budgets its memory up front, code where
an allocation could stall or fail at the wrong moment).  It keeps its per-chunk operands in a
fixed 64 MiB array that the library reserves on each GPU, so it must agree with
kda_chunk_forward_split, which allocates its scratch per call, on every call, including a
second call that finds the previous call's data still in the array.

This file is collected last on purpose, so a run that stops at the first failure has run
every other test before this one.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from gated_delta_rule_26_gb300 import build as kbuild
from gated_delta_rule_26_gb300 import inputs

BF16_REL, BF16_ABS = 2e-2, 5e-2  # the bf16 bar of the parity tests


def _close_to_oracle(got, ref):
    got = got.detach().double().cpu().numpy()
    rel = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-30)
    mx = np.abs(got - ref).max()
    assert rel <= BF16_REL and mx <= BF16_ABS, (rel, mx)


@pytest.mark.gpu
def test_noalloc_split_matches_allocating_split_twice(kda):
    # B*H = 32, T = 4000: 63 chunks (the last one ragged), h0 given.  One chunk of all 32
    # sequences takes 2.4 MB of the 64 MiB array, so the no-alloc call runs segments of 28,
    # 28 and 7 chunks (27, 27 and 9 without hT); the allocating call cuts elsewhere (segments
    # of 18, 18, 18 and 9 chunks on two operand buffers, the carry on a second stream).  Both run the same per-chunk arithmetic and hand the fp32 state
    # across every cut unrounded, so their outputs are identical bit for bit.
    inp = inputs.make(2, 16, 4000, 128, 128, chunk=64, dtype="bf16", seed=31, h0_std=0.1,
                      dt_std=0.1)
    d = inp.to("cuda")
    args = (d.q, d.k, d.v, d.z, d.beta, d.A_log, d.dt_bias, inp.scale, d.h0, 64)
    o_ref, h_ref = kda.chunk_forward(*args, form="split")
    torch.cuda.synchronize()
    for _ in range(2):  # the second call runs on the array the first one left behind
        o, h = kda.chunk_forward(*args, form="split_noalloc")
        torch.cuda.synchronize()
        assert kda.device_status() == 0
        assert torch.equal(o, o_ref)
        assert torch.equal(h, h_ref)
    # without hT the carried state lives in the array too
    o2_ref, _ = kda.chunk_forward(*args, form="split", output_final_state=False)
    o2, _ = kda.chunk_forward(*args, form="split_noalloc", output_final_state=False)
    torch.cuda.synchronize()
    assert kda.device_status() == 0
    assert torch.equal(o2, o2_ref)
    assert torch.equal(o2, o_ref)
    # and against the f64 oracle on three sampled sequences, token by token
    pairs = [(0, 0), (1, 7), (1, 15)]
    bs, hs = [p[0] for p in pairs], [p[1] for p in pairs]
    g = lambda t: t[bs, hs].unsqueeze(0)
    ro, rh = oracle.forward(g(inp.q), g(inp.k), g(inp.v), g(inp.z), g(inp.beta), inp.A_log[hs],
                            inp.dt_bias[hs], inp.scale, g(inp.h0), threads=len(pairs))
    _close_to_oracle(o[bs, hs].unsqueeze(0), ro)
    _close_to_oracle(h[bs, hs].unsqueeze(0), rh)


class _Dims(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("H", ctypes.c_int), ("T", ctypes.c_int),
                ("K", ctypes.c_int), ("V", ctypes.c_int)]


def test_noalloc_rejects_too_many_sequences_on_the_host():
    # more sequences than one chunk each fits in the array: refused before any launch, so the
    # fake (never dereferenced) pointers below are fine and no GPU is needed
    lib = ctypes.CDLL(kbuild.build())
    f = lib.kda_chunk_forward_split_noalloc
    vp = ctypes.c_void_p
    f.argtypes = [vp, ctypes.c_int] + [vp] * 7 + [ctypes.c_float, vp, ctypes.c_int, vp, vp, vp]
    p = vp(1 << 20)
    call = lambda B, H, hT: f(ctypes.byref(_Dims(B, H, 64, 128, 128)), 1, p, p, p, p, p, p, p,
                              0.1, None, 64, p, hT, None)
    assert call(1, 904, p) == -2       # 904 * 74,240 bytes > 64 MiB
    assert call(8, 113, p) == -2       # the same count as B * H
    assert call(1, 481, None) == -2    # without hT: 481 * (74,240 + 65,536) > 64 MiB
