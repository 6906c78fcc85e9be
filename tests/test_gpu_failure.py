"""Failure detection without a GPU fault (GPU only).

Every wait inside the kernels is bounded; when one runs out the kernel
records a status word and unwinds instead of hanging.  Here a one-CTA kernel
waits on an mbarrier that nothing ever arrives at, with a 2 ms limit: the
call must return, report the timeout, and leave the context usable for a
normal attention call afterwards.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import workloads
import tiled_exact_attention_fa2_gb300 as fa2
from parity_util import check_lse, check_o, to_np

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_context_survives():
    lib = fa2.load_library()
    st = ctypes.c_int(-1)
    assert lib.fa2_check_wait_timeout(2000, ctypes.byref(st)) == 0
    assert st.value == 1  # the wait ran out and said so
    # the attention kernels' own status word is untouched and the context works
    assert fa2.fa2_device_status(reset=True) == 0
    x = workloads.make_inputs(1, 2, 150, 64, seed=21)
    g = {k: t.to("cuda:0") for k, t in x.items()}
    o, lse = fa2.fa2_fwd(g["q"], g["k"], g["v"], causal=True)
    torch.cuda.synchronize()
    ref_o, ref_l = oracle.attn_fwd(x["q"], x["k"], x["v"], 1 / np.sqrt(64), True)
    check_o(to_np(o), ref_o)
    check_lse(to_np(lse), ref_l)


def test_bounded_wait_argument_checks():
    lib = fa2.load_library()
    st = ctypes.c_int(0)
    assert lib.fa2_check_wait_timeout(0, ctypes.byref(st)) == 2
    assert lib.fa2_check_wait_timeout(100, None) == 1
