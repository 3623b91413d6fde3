"""The C ABI without a GPU: the library builds, loads and exports every symbol the
header declares, and argument validation refuses bad calls before touching the
device (every call below returns from host-side checks; none launches)."""

import ctypes
import os
import re

import pytest

from virtual_noise_perturbed_gb300 import _lib, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "vn.h")
P = ctypes.c_void_p


@pytest.fixture(scope="module")
def lib():
    build.build()
    return _lib.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(vn_[a-z_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ["vn_perturbed_linear", "vn_weight_gradient", "vn_bias_gradient", "vn_noise_dump"]:
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert name in _lib.SIGNATURES, f"binding lacks {name}"


def test_status_strings(lib):
    for code, name in _lib.STATUS_NAMES.items():
        assert lib.vn_status_string(code).decode().startswith(name)
    assert lib.vn_version() >> 16 == 1


def _dump(lib, seeds, pop, n, out):
    return lib.vn_noise_dump(P(seeds), pop, n, 0, P(out), P(0))


def test_validation_refuses_before_launch(lib):
    fake = 0x1000  # never dereferenced: every call below fails validation first
    assert _dump(lib, fake, -1, 4, fake) == 2                      # VN_ERR_SHAPE
    assert _dump(lib, 0, 4, 4, fake) == 1                          # VN_ERR_NULL
    assert _dump(lib, fake + 4, 4, 4, fake) == 5                   # VN_ERR_ALIGN (seeds)
    assert _dump(lib, fake, 1 << 40, 1 << 40, fake) == 6           # VN_ERR_OVERFLOW
    # gradients: pop >= 1, sigma finite and nonzero
    g = lib.vn_weight_gradient
    assert g(P(fake), P(fake), 0, 4, 4, 0.1, 0, P(fake), P(0)) == 2
    assert g(P(fake), P(fake), 4, 4, 4, 0.0, 0, P(fake), P(0)) == 4
    assert g(P(fake), P(fake), 4, 4, 4, float("nan"), 0, P(fake), P(0)) == 4
    assert g(P(fake), P(fake), 4, 4, 4, 1e300, 0, P(fake), P(0)) == 4
    assert g(P(fake), P(0), 4, 4, 4, 0.1, 0, P(fake), P(0)) == 1
    assert g(P(fake + 2), P(fake), 4, 4, 4, 0.1, 0, P(fake), P(0)) == 5
    assert lib.vn_bias_gradient(P(fake), P(fake), 4, -1, 0.1, 0, P(fake), P(0)) == 2
    # reduce metric: n_params >= 1
    assert lib.vn_reduce_metric(P(fake), P(fake), 4, 0, 0.1, 0, P(fake), P(0)) == 2
    assert lib.vn_reduce_metric(P(fake), P(fake), 4, 8, float("inf"), 0, P(fake), P(0)) == 4
    # forward: dtype rules, shapes, enums
    f = lib.vn_perturbed_linear_ex
    args = lambda **k: dict(dict(x=fake, xd=0, sh=0, w=fake, wd=0, b=0, bd=0, s=fake, pop=2, batch=2,
                                 i=4, o=4, sig=0.1, off=0, y=fake, yd=0, path=0, act=0), **k)

    def call(**k):
        a = args(**k)
        return f(P(a["x"]), a["xd"], a["sh"], P(a["w"]), a["wd"], P(a["b"]), a["bd"], P(a["s"]),
                 a["pop"], a["batch"], a["i"], a["o"], a["sig"], a["off"], P(a["y"]), a["yd"],
                 a["path"], a["act"], P(0))
    assert call(xd=7) == 3                         # unknown dtype
    assert call(xd=1, wd=1, yd=0) == 3             # bf16 x bf16 must give bf16
    assert call(xd=1, wd=0, yd=1) == 3             # mixed gives fp32
    assert call(path=9) == 10                      # unknown path
    assert call(act=5) == 4                        # unknown activation
    assert call(batch=-1) == 2
    assert call(sig=float("nan")) == 4
    assert call(pop=1 << 40, batch=1 << 40) == 6
    assert call(s=0) == 1
    assert call(y=fake + 1) == 5
    assert call(x=0) == 1
    assert call(w=0) == 1


def test_empty_outputs_are_valid_and_launch_nothing(lib):
    assert _dump(lib, 0, 0, 100, 0) == 0
    assert _dump(lib, 0, 100, 0, 0) == 0
    assert lib.vn_weight_gradient(P(0), P(0), 3, 0, 5, 0.1, 0, P(0), P(0)) == 0
    assert lib.vn_reduce_metric(P(0), P(0), 0, 5, 0.1, 0, P(0), P(0)) == 0
    assert lib.vn_perturbed_linear(P(0), 0, 0, P(0), 0, P(0), 0, P(0), 0, 4, 4, 4, 0.1, 0,
                                   P(0), 0, P(0)) == 0


def test_mlp_validation_refuses_before_launch(lib):
    fake = 0x1000
    I64, U64, VP = ctypes.c_int64, ctypes.c_uint64, ctypes.c_void_p

    def call(n=2, dims=(4, 8, 2), w=(fake, fake), b=None, offs=(0, 40), x=fake, xd=0, s=fake,
             pop=3, batch=1, sig=0.1, act=1, y=fake):
        cd = (I64 * len(dims))(*dims)
        cw = (VP * len(w))(*w)
        cb = None if b is None else (VP * len(b))(*b)
        co = (U64 * len(offs))(*offs)
        return lib.vn_perturbed_mlp(P(x), xd, 0, n, cd, cw, cb, co, P(s), pop, batch, sig, act,
                                    P(y), P(0))
    assert call(xd=5) == 3                        # unknown x dtype
    assert call(act=9) == 4                       # unknown activation
    assert call(n=0) == 2                         # no layers
    assert call(n=9, dims=(4,) * 10, w=(fake,) * 9, offs=(0,) * 9) == 2   # more than 8 layers
    assert call(batch=9) == 2                     # batch above 8
    assert call(dims=(4, -8, 2)) == 2
    assert call(sig=float("inf")) == 4
    assert call(w=(fake, 0)) == 1                 # a layer with weights needs a pointer
    assert call(w=(fake + 2, fake)) == 5          # fp32 weights 4-byte aligned
    assert call(b=(fake, fake + 1)) == 5
    assert call(s=0) == 1
    assert call(y=fake + 2) == 5
    assert call(x=0) == 1
    assert call(pop=1 << 40, batch=8, dims=(4, 8, 1 << 30)) == 6
    assert call(pop=0, s=0, y=0, x=0) == 0        # empty output: valid, nothing launched
    assert call(dims=(4, 8, 0), y=0) == 0


def test_ranks_and_update_validation(lib):
    fake = 0x1000
    assert lib.vn_centered_ranks(P(fake), -1, P(fake + 64), P(0)) == 2          # negative pop
    assert lib.vn_centered_ranks(P(fake), 1 << 31, P(fake + 64), P(0)) == 2     # pop >= 2^31
    assert lib.vn_centered_ranks(P(0), 0, P(0), P(0)) == 0                      # empty: nothing launched
    assert lib.vn_centered_ranks(P(0), 4, P(fake), P(0)) == 1
    assert lib.vn_centered_ranks(P(fake + 2), 4, P(fake + 64), P(0)) == 5
    assert lib.vn_centered_ranks(P(fake), 4, P(fake + 8), P(0)) == 4            # overlapping in/out
    assert lib.vn_es_update(P(fake), P(fake), -1, 0.1, P(0)) == 2
    assert lib.vn_es_update(P(fake), P(fake), 4, float("inf"), P(0)) == 4
    assert lib.vn_es_update(P(0), P(0), 0, 0.1, P(0)) == 0
    assert lib.vn_es_update(P(0), P(fake), 4, 0.1, P(0)) == 1
    assert lib.vn_es_update(P(fake), P(fake + 1), 4, 0.1, P(0)) == 5


def test_noise_kind_validation(lib):
    fake = 0x1000
    assert lib.vn_noise_dump_ex(P(fake), 1, 4, 0, 7, P(fake), P(0)) == 4        # unknown kind
    assert lib.vn_noise_dump_ex(P(fake), -1, 4, 0, 1, P(fake), P(0)) == 2
    assert lib.vn_noise_dump_ex(P(0), 0, 4, 0, 1, P(0), P(0)) == 0               # empty
    assert lib.vn_gradient_ex(P(fake), P(fake), 1, 4, 0.1, 0, 2, P(fake), P(0)) == 4
    assert lib.vn_gradient_ex(P(fake), P(fake), 0, 4, 0.1, 0, 1, P(fake), P(0)) == 2
    assert lib.vn_gradient_ex(P(fake), P(fake), 4, 4, 0.0, 0, 1, P(fake), P(0)) == 4


def test_gradient_update_validation(lib):
    fake = 0x1000
    gu = lib.vn_gradient_update
    # (fitness, seeds, pop, n, sigma, offset, kind, lr, grad, theta, stream)
    assert gu(P(fake), P(fake), 4, 4, 0.1, 0, 0, 0.1, P(fake), P(0), P(0)) == 1       # theta NULL
    assert gu(P(fake), P(fake), 4, 4, 0.1, 0, 0, float("nan"), P(fake), P(fake + 64), P(0)) == 4
    assert gu(P(fake), P(fake), 4, 4, 0.0, 0, 0, 0.1, P(fake), P(fake + 64), P(0)) == 4  # sigma 0
    assert gu(P(fake), P(fake), 0, 4, 0.1, 0, 0, 0.1, P(fake), P(fake + 64), P(0)) == 2  # pop 0
    assert gu(P(fake), P(fake), 4, 4, 0.1, 0, 3, 0.1, P(fake), P(fake + 64), P(0)) == 4  # kind
    assert gu(P(fake), P(fake), 4, 4, 0.1, 0, 0, 0.1, P(fake), P(fake + 66), P(0)) == 5  # theta align
    assert gu(P(fake), P(fake), 4, 4, 0.1, 0, 0, 0.1, P(fake), P(fake + 8), P(0)) == 4   # theta overlaps grad
    assert gu(P(fake), P(fake), 4, 0, 0.1, 0, 0, 0.1, P(0), P(0), P(0)) == 0             # empty


def test_mlp_ex_refuses_unknown_noise_kind(lib):
    fake = 0x1000
    dims = (ctypes.c_int64 * 2)(4, 4)
    ptrs = (ctypes.c_void_p * 1)(fake)
    offs = (ctypes.c_uint64 * 1)(0)
    f = lib.vn_perturbed_mlp_ex
    assert f(P(fake), 0, 0, 1, dims, ptrs, None, offs, P(fake), 4, 1, 0.1, 1, 2, P(fake), P(0)) == 4
    assert f(P(fake), 0, 0, 1, dims, ptrs, None, offs, P(fake), 4, 9, 0.1, 1, 1, P(fake), P(0)) == 2


def test_linear_kind_refuses_unknown_noise_kind(lib):
    fake = 0x1000
    f = lib.vn_perturbed_linear_kind
    # (x, x_dt, shared, w, w_dt, b, b_dt, seeds, pop, batch, in, out, sigma, offset, y, y_dt, path, act, kind, s)
    assert f(P(fake), 0, 0, P(fake), 0, P(0), 0, P(fake), 4, 1, 8, 8, 0.1, 0, P(fake), 0, 0, 0, 5, P(0)) == 4
    assert f(P(fake), 0, 0, P(fake), 0, P(0), 0, P(fake), -1, 1, 8, 8, 0.1, 0, P(fake), 0, 0, 0, 1, P(0)) == 2


def test_testhook_checks_like_the_tensor_core_call(lib):
    """The bounded-wait test hook runs the same checks as vn_perturbed_linear_kind,
    with its real population: a misaligned or overlapping output is refused before
    any device query or launch."""
    fake = 0x10000
    x, w, b, s = fake + 0x1000, fake + 0x2000, fake + 0x3000, fake + 0x4000
    hook = lib.vn_testhook_linear_tc_withhold

    def call(y, pop=2, bias=b, stage=0, ms=50.0, seeds=s):
        # bf16 x, w, b and y: (x, 1, 0, w, 1, b, 1, seeds, pop, batch 2, in 8, out 4, sigma, offset, y, 1, ...)
        return hook(P(x), 1, 0, P(w), 1, P(bias), 1, P(seeds), pop, 2, 8, 4, 0.1, 0, P(y), 1, stage, ms, P(0))
    assert call(fake + 0x5001) == 5          # y misaligned for bf16: VN_ERR_ALIGN
    assert call(x + 16) == 4                 # y over x: VN_ERR_VALUE
    assert call(w + 2) == 4                  # y over w
    assert call(s + 8) == 4                  # y over the seeds
    assert call(fake + 0x5000, seeds=s + 4) == 5   # seeds misaligned
    assert call(fake + 0x5000, pop=0) == 2   # nothing to withhold an arrive in: VN_ERR_SHAPE
    assert call(fake + 0x5000, stage=-1) == 4
    assert call(fake + 0x5000, ms=0.0) == 4
    assert hook(P(x), 1, 0, P(w), 0, P(b), 1, P(s), 2, 2, 8, 4, 0.1, 0, P(fake + 0x5000), 0, 0, 50.0,
                P(0)) == 3                   # fp32 W: the hook has bf16 W and Y only


def test_outputs_overlapping_inputs_are_refused(lib):
    """Every call refuses an output that shares bytes with one of its inputs (or
    with its other output) before anything is launched: VN_ERR_VALUE."""
    fake = 0x10000
    f_, s_, g_ = fake, fake + 0x100, fake + 0x200            # fitness, seeds, a free area
    # dump: 4 x 4 floats over the 4 seeds
    assert lib.vn_noise_dump(P(s_), 4, 4, 0, P(s_ + 16), P(0)) == 4
    # gradients: grad over fitness, grad over seeds
    assert lib.vn_weight_gradient(P(f_), P(s_), 4, 2, 2, 0.1, 0, P(f_ + 12), P(0)) == 4
    assert lib.vn_bias_gradient(P(f_), P(s_), 4, 4, 0.1, 0, P(s_ + 28), P(0)) == 4
    assert lib.vn_gradient_ex(P(f_), P(s_), 4, 4, 0.1, 0, 1, P(s_ - 12), P(0)) == 4
    # gradient + update: theta over fitness, over seeds, over grad
    gu = lib.vn_gradient_update
    assert gu(P(f_), P(s_), 4, 4, 0.1, 0, 0, 0.1, P(g_), P(f_ + 4), P(0)) == 4
    assert gu(P(f_), P(s_), 4, 4, 0.1, 0, 0, 0.1, P(g_), P(s_ + 16), P(0)) == 4
    assert gu(P(f_), P(s_), 4, 4, 0.1, 0, 0, 0.1, P(g_), P(g_ + 12), P(0)) == 4
    # metric: fitness over center (8 floats), over seeds
    assert lib.vn_reduce_metric(P(g_), P(s_), 4, 8, 0.1, 0, P(g_ + 28), P(0)) == 4
    assert lib.vn_reduce_metric(P(g_), P(s_), 4, 8, 0.1, 0, P(s_ + 24), P(0)) == 4
    # forward: y (2 x 2 x 4 floats) over x, w, b and seeds
    x, w, b, s = fake + 0x1000, fake + 0x2000, fake + 0x3000, fake + 0x4000

    def lin(y, bias=b):
        return lib.vn_perturbed_linear(P(x), 0, 0, P(w), 0, P(bias), 0, P(s), 2, 2, 4, 4, 0.1, 0,
                                       P(y), 0, P(0))
    assert lin(x + 60) == 4          # the last float of x
    assert lin(w - 60) == 4          # y's last float is w's first
    assert lin(b + 8) == 4
    assert lin(s + 12) == 4
    # chain forward: y over a layer's weights, its bias, x
    dims = (ctypes.c_int64 * 3)(4, 4, 4)
    ws = (ctypes.c_void_p * 2)(w, w + 0x100)
    bs = (ctypes.c_void_p * 2)(b, b + 0x100)
    offs = (ctypes.c_uint64 * 2)(0, 20)

    def mlp(y, bias=None):
        return lib.vn_perturbed_mlp(P(x), 0, 0, 2, dims, ws, bias, offs, P(s), 2, 1, 0.1, 1, P(y), P(0))
    assert mlp(w + 0x100 + 60) == 4  # the second layer's last weight
    assert mlp(b + 0x100, bs) == 4   # the second layer's bias
    assert mlp(x + 4) == 4
    # parameter step and ranks
    assert lib.vn_es_update(P(g_), P(g_ + 8), 4, 0.1, P(0)) == 4
    assert lib.vn_centered_ranks(P(g_), 4, P(g_ + 12), P(0)) == 4


def test_binding_requires_one_device_per_call():
    """The binding runs each call with its tensors' device made current, and refuses
    a call whose tensors sit on different devices."""
    import torch
    from virtual_noise_perturbed_gb300 import api
    with pytest.raises(ValueError, match="share a device"):
        api._device(torch.empty(1), torch.empty(1, device="meta"))
    assert api._device(torch.empty(1), None, torch.empty(2)) == torch.device("cpu")


def test_concurrent_builds_take_turns_and_build_once(monkeypatch, tmp_path):
    """build() holds a file lock around compile and link: callers that start together
    (the ranks of one job) build one at a time, and one that finds the library current
    after waiting does not build again. The compile step is a stand-in here."""
    import threading
    import time

    from virtual_noise_perturbed_gb300 import build as b
    monkeypatch.setattr(b, "BUILD", str(tmp_path))
    state = {"current": False, "spans": []}
    monkeypatch.setattr(b, "up_to_date", lambda: state["current"])

    def compile_step(verbose, extra_flags):
        t0 = time.monotonic()
        time.sleep(0.2)
        state["spans"].append((t0, time.monotonic()))

    monkeypatch.setattr(b, "_compile_and_link", compile_step)
    threads = [threading.Thread(target=b.build, kwargs={"force": True}) for _ in range(3)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    spans = sorted(state["spans"])
    assert len(spans) == 3                                    # forced: each builds, in turn
    assert all(a[1] <= c[0] for a, c in zip(spans, spans[1:]))

    state["spans"].clear()

    def compile_once(verbose, extra_flags):
        compile_step(verbose, extra_flags)
        state["current"] = True

    monkeypatch.setattr(b, "_compile_and_link", compile_once)
    threads = [threading.Thread(target=b.build) for _ in range(3)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert len(state["spans"]) == 1                           # the others found it current


def test_binding_output_buffers_are_checked():
    """``out=`` buffers must be contiguous float32 of the result's shape on the call's device."""
    import torch
    from virtual_noise_perturbed_gb300 import api
    cpu = torch.device("cpu")
    buf = torch.zeros(3, 4)
    assert api._out(buf, (3, 4), cpu) is buf
    assert api._out(None, (2,), cpu).shape == (2,)
    for bad in (torch.zeros(4, 3), torch.zeros(3, 4, dtype=torch.float64), torch.zeros(4, 3).t(),
                torch.zeros(3, 4, device="meta")):
        with pytest.raises(ValueError):
            api._out(bad, (3, 4), cpu)
