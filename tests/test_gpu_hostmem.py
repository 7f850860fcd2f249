"""Page-locked host tensors as inputs and outputs (zero copy: the kernel
reads and writes them over the host link with plain loads and stores).
Results must equal the device-memory results bit for bit (the arithmetic is
the same; only the staging differs) and match the oracle."""
import numpy as np
import pytest
import torch

import oracle
from linear_recurrence_scan_gb300 import synthetic

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def built():
    from linear_recurrence_scan_gb300 import build
    build.build()


def L():
    import linear_recurrence_scan_gb300 as lib
    return lib


def pinned(a):
    return None if a is None else torch.from_numpy(np.ascontiguousarray(a)).pin_memory()


def device(a):
    return None if a is None else torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def same(host_out, dev_out, what):
    torch.cuda.synchronize()
    assert not host_out.is_cuda and host_out.is_pinned(), what
    assert torch.equal(host_out, dev_out.cpu()), what


@pytest.mark.parametrize("shape", [(8, 128), (4096, 1024), (3, 3000), (64, 1 << 15), (5, 37)],
                         ids=["8x128", "4096x1024", "3x3000", "64x32768", "5x37"])
def test_gae_and_returns_zero_copy(shape):
    N, T = shape
    b = synthetic.returns_batch(N, T, 9, 81)
    keys = ("rewards", "values", "terminateds")
    h = L().compute_gae_and_returns(*(pinned(b[k]) for k in keys), None, 0.99, 0.95, None,
                                    pinned(b["last_value"]))
    d = L().compute_gae_and_returns(*(device(b[k]) for k in keys), None, 0.99, 0.95, None,
                                    device(b["last_value"]))
    for x, y, w in zip(h, d, ("advantages", "lambda returns", "discounted returns")):
        same(x, y, w)
    ref = oracle.gae(b["rewards"], b["values"], b["terminateds"], None, 0.99, 0.95, None,
                     b["last_value"])
    err = np.abs(h[0].double().numpy() - ref)
    assert (err <= 1e-4 + 1e-5 * np.abs(ref)).all()


def test_vtrace_zero_copy_mixed_residency():
    """Inputs partly on the device, partly pinned on the host."""
    b = synthetic.vtrace_batch(16, 3000, 9, 82)
    args_h = [pinned(b[k]) if i % 2 else device(b[k]) for i, k in enumerate(
        ("log_pi_target", "log_pi_behavior", "values", "rewards", "terminateds", "truncateds"))]
    args_d = [device(b[k]) for k in
              ("log_pi_target", "log_pi_behavior", "values", "rewards", "terminateds", "truncateds")]
    vs_h, adv_h = L().compute_vtrace(*args_h, 0.99, 1.0, 1.0, device(b["bootstrap_values"]))
    vs_d, adv_d = L().compute_vtrace(*args_d, 0.99, 1.0, 1.0, device(b["bootstrap_values"]))
    torch.cuda.synchronize()
    assert torch.equal(vs_h.cpu(), vs_d.cpu()) and torch.equal(adv_h.cpu(), adv_d.cpu())


def test_retrace_actions_zero_copy():
    b = synthetic.retrace_actions_batch(8, 3000, 4, 9, 83)
    keys = ("action_probs_target", "action_probs_behavior", "q_values", "next_q_values_all",
            "actions", "rewards", "terminateds")
    h = L().compute_retrace(*(pinned(b[k]) for k in keys), None, 0.99, 0.95)
    d = L().compute_retrace(*(device(b[k]) for k in keys), None, 0.99, 0.95)
    same(h[0], d[0], "retrace targets")
    same(h[1], d[1], "retrace advantages")


def test_compact_and_normalized_zero_copy():
    b = synthetic.returns_batch(64, 2048, 9, 84)
    rb = torch.from_numpy(b["rewards"]).to(torch.bfloat16)
    vb = torch.from_numpy(b["values"]).to(torch.bfloat16)
    tb = torch.from_numpy(b["terminateds"]).to(torch.uint8)
    last = torch.from_numpy(b["last_value"])
    h = L().compute_gae(rb.pin_memory(), vb.pin_memory(), tb.pin_memory(), None, 0.99, 0.95, None,
                        last.pin_memory(), out_dtype=torch.bfloat16)
    d = L().compute_gae(rb.to(DEV), vb.to(DEV), tb.to(DEV), None, 0.99, 0.95, None, last.to(DEV),
                        out_dtype=torch.bfloat16)
    same(h, d, "compact gae")
    keys = ("rewards", "values", "terminateds")
    hn = L().compute_gae_normalized(*(pinned(b[k]) for k in keys), None, 0.99, 0.95, None,
                                    pinned(b["last_value"]))
    dn = L().compute_gae_normalized(*(device(b[k]) for k in keys), None, 0.99, 0.95, None,
                                    device(b["last_value"]))
    same(hn[0], dn[0], "normalised advantages")
    same(hn[1], dn[1], "lambda returns")


def test_plain_cpu_tensors_are_rejected():
    x = torch.zeros(2, 4)
    with pytest.raises(ValueError, match="pinned"):
        L().compute_gae(x, x, x)


def test_strided_pinned_inputs_stay_page_locked():
    """Pinned inputs whose strides differ are re-laid out; the copies must
    stay page-locked (the kernel reads host tensors in place)."""
    N, T = 8, 3000
    b = synthetic.returns_batch(N, T, 9, 85)
    r = pinned(b["rewards"])
    wide = torch.zeros((N, T + 8), dtype=torch.float32).pin_memory()
    wide[:, :T] = torch.from_numpy(b["values"])
    v = wide[:, :T]                               # row stride T + 8, the others T
    term = pinned(b["terminateds"])
    last = torch.zeros(2 * N, dtype=torch.float32).pin_memory()
    last[::2] = torch.from_numpy(b["last_value"])
    h = L().compute_gae(r, v, term, None, 0.99, 0.95, None, last[::2])   # strided [N] vector too
    d = L().compute_gae(device(b["rewards"]), device(b["values"]), device(b["terminateds"]), None, 0.99, 0.95,
                        None, device(b["last_value"]))
    same(h, d, "strided pinned gae")


def test_pageable_memory_through_the_c_abi():
    """Pageable host arrays passed to the C ABI: read and written in place on
    a device that reads pageable memory (equal to the device path bit for
    bit), refused with RLSCAN_ERR_MEMORY (output untouched) on one that
    does not.  A page-locked host workspace is refused."""
    import ctypes
    from linear_recurrence_scan_gb300 import _native
    lib = _native.lib()
    N, T = 8, 3000
    b = synthetic.returns_batch(N, T, 9, 86)
    r, v, term = (np.ascontiguousarray(b[k], dtype=np.float32) for k in ("rewards", "values", "terminateds"))
    last = np.ascontiguousarray(b["last_value"], dtype=np.float32)
    out = np.zeros((N, T), dtype=np.float32)
    wsn = lib.rlscan_workspace_bytes(N, T)
    ws = torch.zeros(wsn, dtype=torch.uint8, device=DEV)
    s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    st = lib.rlscan_gae(r.ctypes.data, v.ctypes.data, term.ctypes.data, None, None, last.ctypes.data, N, T, T,
                        0.99, 0.95, out.ctypes.data, ws.data_ptr(), wsn, s)
    torch.cuda.synchronize()
    if st == 0:
        d = L().compute_gae(device(b["rewards"]), device(b["values"]), device(b["terminateds"]), None, 0.99, 0.95,
                            None, device(b["last_value"]))
        assert np.array_equal(out, d.cpu().numpy())
    else:
        assert _native.STATUS[st] == "RLSCAN_ERR_MEMORY", _native.STATUS.get(st, st)
        assert not out.any()
    host_ws = torch.zeros(wsn, dtype=torch.uint8).pin_memory()
    rp, vp, tp = (pinned(b[k]) for k in ("rewards", "values", "terminateds"))
    st = lib.rlscan_gae(rp.data_ptr(), vp.data_ptr(), tp.data_ptr(), None, None, pinned(last).data_ptr(), N, T, T,
                        0.99, 0.95, pinned(out).data_ptr(), host_ws.data_ptr(), wsn, s)
    torch.cuda.synchronize()
    assert _native.STATUS[st] == "RLSCAN_ERR_WORKSPACE"


def test_pinned_copies_outlive_the_kernel_that_reads_them():
    """A strided pinned input is re-laid out into a page-locked copy that the
    kernel reads over the host link after the call has returned.  The copy
    must stay referenced until the stream has passed the call: right after
    each call, fresh pinned blocks of the same size are allocated and
    overwritten (what a freed copy's block would be handed to), and every
    result must still equal the device-memory one.  Once the stream has
    synchronised, the next call releases the copies."""
    import linear_recurrence_scan_gb300.api as api
    N, T = 256, 4096
    b = synthetic.returns_batch(N, T, 11, 86)
    d = L().compute_gae(device(b["rewards"]), device(b["values"]), device(b["terminateds"]), None, 0.99, 0.95,
                        None, device(b["last_value"]))
    outs, junk = [], []
    for _ in range(4):
        wide = torch.zeros((N, T + 4), dtype=torch.float32).pin_memory()
        wide[:, :T] = torch.from_numpy(b["values"])
        v = wide[:, :T]                          # row stride T + 4: every input is copied
        outs.append(L().compute_gae(pinned(b["rewards"]), v, pinned(b["terminateds"]), None, 0.99, 0.95, None,
                                    pinned(b["last_value"])))
        del wide, v
        for _ in range(3):                       # blocks a released copy could be handed to
            j = torch.empty((N, T), dtype=torch.float32).pin_memory()
            j.fill_(float("nan"))
            junk.append(j)
    for i, h in enumerate(outs):
        same(h, d, f"pinned copies, call {i}")
    torch.cuda.synchronize()
    L().compute_gae(device(b["rewards"]), device(b["values"]), device(b["terminateds"]), None, 0.99, 0.95,
                    None, device(b["last_value"]))
    assert len(api._held) == 0
