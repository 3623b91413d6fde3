"""Python API with the EvoX page's names and signatures, over the C ABI.

EvoX API page "evox.triton_kernels.kernels.virtual_noise": API entries
``virtual_perturbed_linear``, ``virtual_weight_gradient``,
``virtual_bias_gradient``, ``virtual_reduce_metric``, ``compute_offsets`` and
the ``_cpu_normal_noise`` contract (here ``noise_dump``).

These functions only check and marshal arguments (contiguity, integer seeds
widened to int64, output allocation) and call ``libvn.so`` on the current
CUDA stream; all arithmetic runs in the library's kernels. Tensors must be on
a CUDA device; there is no CPU path.
"""

from __future__ import annotations

import ctypes
import math
from typing import Optional, Sequence

import torch

from . import _lib
from ._lib import VNError, check, load

_DT = {torch.float32: _lib.VN_F32, torch.bfloat16: _lib.VN_BF16}
_PATHS = {"auto": _lib.VN_PATH_AUTO, "ffma": _lib.VN_PATH_FFMA, "tc": _lib.VN_PATH_TC}
_ACTS = {None: _lib.VN_ACT_NONE, "none": _lib.VN_ACT_NONE, "tanh": _lib.VN_ACT_TANH}
_NOISE = {"uniform": _lib.VN_NOISE_UNIFORM, "gaussian": _lib.VN_NOISE_GAUSSIAN}
_M64 = (1 << 64) - 1


def _cuda(t: torch.Tensor, name: str) -> torch.Tensor:
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (the library has no CPU path)")
    return t.contiguous()


def _dt(t: torch.Tensor, name: str) -> int:
    try:
        return _DT[t.dtype]
    except KeyError:
        raise TypeError(f"{name}: dtype {t.dtype} is not supported (float32 or bfloat16)") from None


def _seeds(seeds: torch.Tensor) -> torch.Tensor:
    seeds = _cuda(seeds, "seeds")
    if seeds.dim() != 1:
        raise ValueError("seeds must be 1-D")
    if seeds.dtype not in (torch.int64, torch.int32, torch.int16, torch.int8, torch.uint8):
        raise TypeError(f"seeds must be an integer tensor, got {seeds.dtype}")
    return seeds.to(torch.int64)


def _stream(t: torch.Tensor) -> ctypes.c_void_p:
    return ctypes.c_void_p(torch.cuda.current_stream(t.device).cuda_stream)


def _ptr(t: Optional[torch.Tensor]) -> ctypes.c_void_p:
    return ctypes.c_void_p(0 if t is None or t.numel() == 0 else t.data_ptr())


def _out(out: Optional[torch.Tensor], shape, device: torch.device) -> torch.Tensor:
    """The caller's float32 output buffer, checked (shape, dtype, layout, device), or a new one."""
    shape = tuple(int(d) for d in shape)
    if out is None:
        return torch.empty(shape, dtype=torch.float32, device=device)
    if not isinstance(out, torch.Tensor) or tuple(out.shape) != shape or out.dtype != torch.float32 \
            or not out.is_contiguous() or out.device != device:
        raise ValueError(f"out must be a contiguous float32 tensor of shape {shape} on {device}")
    return out


def _device(*tensors: Optional[torch.Tensor]) -> torch.device:
    """The one device every tensor of a call is on. The library launches on the
    current CUDA device, so each call runs with this device made current."""
    devices = {t.device for t in tensors if t is not None}
    if len(devices) != 1:
        raise ValueError(f"the tensors of one call must share a device, got {sorted(map(str, devices))}")
    return devices.pop()


def virtual_perturbed_linear(x: torch.Tensor, weight: torch.Tensor, bias: Optional[torch.Tensor],
                             seeds: torch.Tensor, sigma: float, offset: int, *,
                             activation: Optional[str] = None, path: str = "auto",
                             out: Optional[torch.Tensor] = None, noise: str = "uniform",
                             check_status: bool = False) -> torch.Tensor:
    """Y[i] = X[i] @ (W + sigma*N_i)^T + (b + sigma*nb_i), shape (pop, batch, out).

    x is (batch, in) (shared by every individual) or (pop, batch, in). The
    result dtype is torch.result_type(x, weight). ``activation="tanh"`` applies
    tanh to Y in the kernel's epilogue; ``path`` forces "ffma" or "tc"; ``noise="gaussian"``
    perturbs with the Box-Muller variant (``vn_perturbed_linear_kind``).

    The launch is asynchronous. On the tensor-core path every on-chip barrier wait
    is bounded (4 s); a wait that runs out stops the kernel with part of Y unwritten
    and records VN_ERR_TIMEOUT on the device, which only ``device_status()`` reports.
    So Y from that path is valid once ``device_status()`` has returned without
    raising; ``check_status=True`` makes that call here (it synchronises the stream)."""
    lib = load()
    x = _cuda(x, "x")
    weight = _cuda(weight, "weight")
    seeds = _seeds(seeds)
    if weight.dim() != 2:
        raise ValueError("weight must be (out_features, in_features)")
    out_f, in_f = weight.shape
    pop = seeds.numel()
    if x.dim() == 2:
        shared, batch = 1, x.shape[0]
    elif x.dim() == 3:
        if x.shape[0] != pop:
            raise ValueError(f"x has {x.shape[0]} individuals but there are {pop} seeds")
        shared, batch = 0, x.shape[1]
    else:
        raise ValueError("x must be (batch, in) or (pop, batch, in)")
    if x.shape[-1] != in_f:
        raise ValueError(f"x has {x.shape[-1]} features, weight expects {in_f}")
    if bias is not None:
        bias = _cuda(bias, "bias")
        if bias.shape != (out_f,):
            raise ValueError(f"bias must have shape ({out_f},)")
    ydt = torch.bfloat16 if (x.dtype == torch.bfloat16 and weight.dtype == torch.bfloat16) else torch.float32
    if out is None:
        out = torch.empty((pop, batch, out_f), dtype=ydt, device=x.device)
    elif out.shape != (pop, batch, out_f) or out.dtype != ydt or not out.is_contiguous():
        raise ValueError("out has the wrong shape, dtype or layout")
    if activation not in _ACTS or path not in _PATHS:
        raise ValueError("activation must be None/'tanh'; path 'auto'/'ffma'/'tc'")
    if noise not in _NOISE:
        raise ValueError("noise must be 'uniform' or 'gaussian'")
    with torch.cuda.device(_device(x, weight, bias, seeds, out)):
        st = lib.vn_perturbed_linear_kind(
            _ptr(x), _dt(x, "x"), shared, _ptr(weight), _dt(weight, "weight"),
            _ptr(bias), _dt(bias, "bias") if bias is not None else 0,
            _ptr(seeds), pop, batch, in_f, out_f, float(sigma), int(offset) & _M64,
            _ptr(out), _DT[ydt], _PATHS[path], _ACTS[activation], _NOISE[noise], _stream(x))
        check(st, "vn_perturbed_linear")
        if check_status:
            device_status(x.device)
    return out


def virtual_perturbed_mlp(x: torch.Tensor, weights: Sequence[torch.Tensor],
                          biases: Optional[Sequence[Optional[torch.Tensor]]], seeds: torch.Tensor,
                          sigma: float, offsets: Optional[Sequence[int]] = None, *,
                          activation: Optional[str] = "tanh",
                          out: Optional[torch.Tensor] = None, noise: str = "uniform") -> torch.Tensor:
    """A chain of perturbed linear layers in one launch (fp32 weights, batch <= 8).
    ``noise="gaussian"`` perturbs with the Box-Muller variant of the noise
    (``vn_perturbed_mlp_ex``), the counterpart of the Gaussian gradient.

    Layer l computes ``act(h @ (W_l + sigma*N_{i,l})^T + b_l + sigma*nb_{i,l})``
    with the activation on every layer but the last. ``offsets`` are the weight
    blocks' offsets; by default those of ``compute_offsets`` over
    (W_0, b_0, W_1, b_1, ...) -- so layer l's bias noise sits right after its
    weights, as in ``virtual_perturbed_linear``. x is (batch, in) or
    (pop, batch, in); the result is fp32 (pop, batch, out_last)."""
    lib = load()
    x = _cuda(x, "x")
    seeds = _seeds(seeds)
    weights = [_cuda(w, f"weights[{l}]") for l, w in enumerate(weights)]
    n = len(weights)
    if n == 0:
        raise ValueError("at least one layer is needed")
    if biases is None:
        biases = [None] * n
    if len(biases) != n:
        raise ValueError("one bias (or None) per layer")
    dims = [weights[0].shape[1]] + [w.shape[0] for w in weights]
    for l, w in enumerate(weights):
        if w.dim() != 2 or w.shape[1] != dims[l] or w.dtype != torch.float32:
            raise ValueError(f"weights[{l}] must be float32 ({dims[l + 1]}, {dims[l]})")
    biases = [None if b is None else _cuda(b, f"biases[{l}]") for l, b in enumerate(biases)]
    for l, b in enumerate(biases):
        if b is not None and (b.shape != (dims[l + 1],) or b.dtype != torch.float32):
            raise ValueError(f"biases[{l}] must be float32 ({dims[l + 1]},)")
    if offsets is None:
        shapes = []
        for l in range(n):
            shapes += [(dims[l + 1], dims[l]), (dims[l + 1],)]
        offsets = compute_offsets(shapes)[0::2]
    if len(offsets) != n:
        raise ValueError("one offset per layer")
    pop = seeds.numel()
    if x.dim() == 2:
        shared, batch = 1, x.shape[0]
    elif x.dim() == 3:
        if x.shape[0] != pop:
            raise ValueError(f"x has {x.shape[0]} individuals but there are {pop} seeds")
        shared, batch = 0, x.shape[1]
    else:
        raise ValueError("x must be (batch, in) or (pop, batch, in)")
    if x.shape[-1] != dims[0]:
        raise ValueError(f"x has {x.shape[-1]} features, the first layer expects {dims[0]}")
    if activation not in _ACTS:
        raise ValueError("activation must be None or 'tanh'")
    if noise not in _NOISE:
        raise ValueError("noise must be 'uniform' or 'gaussian'")
    if out is None:
        out = torch.empty((pop, batch, dims[-1]), dtype=torch.float32, device=x.device)
    elif out.shape != (pop, batch, dims[-1]) or out.dtype != torch.float32 or not out.is_contiguous():
        raise ValueError("out has the wrong shape, dtype or layout")
    c_dims = (ctypes.c_int64 * (n + 1))(*dims)
    c_w = (ctypes.c_void_p * n)(*[_ptr(w).value for w in weights])
    c_b = (ctypes.c_void_p * n)(*[_ptr(b).value for b in biases])
    c_off = (ctypes.c_uint64 * n)(*[int(o) & _M64 for o in offsets])
    with torch.cuda.device(_device(x, seeds, out, *weights, *biases)):
        st = lib.vn_perturbed_mlp_ex(_ptr(x), _dt(x, "x"), shared, n, c_dims, c_w, c_b, c_off,
                                     _ptr(seeds), pop, batch, float(sigma), _ACTS[activation],
                                     _NOISE[noise], _ptr(out), _stream(x))
    check(st, "vn_perturbed_mlp_ex")
    return out


def _fitness(fitness: torch.Tensor, pop_size: int, seeds: torch.Tensor) -> torch.Tensor:
    fitness = _cuda(fitness, "fitness").reshape(-1).to(torch.float32)
    if fitness.numel() != pop_size or seeds.numel() != pop_size:
        raise ValueError(f"pop_size={pop_size} but {seeds.numel()} seeds and "
                         f"{fitness.numel()} fitness values")
    return fitness


def virtual_weight_gradient(fitness: torch.Tensor, seeds: torch.Tensor, weight_shape: Sequence[int],
                            sigma: float, pop_size: int, offset: int, *,
                            out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """grad[j, k] = sum_i fitness_i * N_i[j, k] / (pop_size * sigma), fp32, weight_shape
    (written into ``out`` when given)."""
    lib = load()
    seeds = _seeds(seeds)
    fitness = _fitness(fitness, pop_size, seeds)
    out_f, in_f = (int(d) for d in weight_shape)
    dev = _device(fitness, seeds)
    g = _out(out, (out_f, in_f), dev)
    with torch.cuda.device(dev):
        st = lib.vn_weight_gradient(_ptr(fitness), _ptr(seeds), pop_size, out_f, in_f, float(sigma),
                                    int(offset) & _M64, _ptr(g), _stream(g))
    check(st, "vn_weight_gradient")
    return g


def virtual_bias_gradient(fitness: torch.Tensor, seeds: torch.Tensor, bias_shape: Sequence[int],
                          sigma: float, pop_size: int, offset: int, *,
                          out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """grad[j] = sum_i fitness_i * nb_i[j] / (pop_size * sigma); ``offset`` points at the bias
    region (written into ``out`` when given)."""
    lib = load()
    seeds = _seeds(seeds)
    fitness = _fitness(fitness, pop_size, seeds)
    (out_f,) = (int(d) for d in bias_shape)
    dev = _device(fitness, seeds)
    g = _out(out, (out_f,), dev)
    with torch.cuda.device(dev):
        st = lib.vn_bias_gradient(_ptr(fitness), _ptr(seeds), pop_size, out_f, float(sigma),
                                  int(offset) & _M64, _ptr(g), _stream(g))
    check(st, "vn_bias_gradient")
    return g


def virtual_flat_gradient(fitness: torch.Tensor, seeds: torch.Tensor, n_params: int, sigma: float,
                          pop_size: int, offset: int = 0, *, noise: str = "uniform",
                          out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """grad[t] = sum_i fitness_i * PRNG(seed_i, offset + t) / (pop_size * sigma), t < n_params.

    With parameter blocks laid out by ``compute_offsets`` (weights then bias, one
    block after another), this is the gradient of every block in one launch:
    block b's gradient is ``grad[offsets[b] : offsets[b] + numel_b]`` reshaped to the
    block's shape, equal (up to the order of the fp32 sums) to
    ``virtual_weight_gradient`` / ``virtual_bias_gradient`` on that block.
    ``noise="gaussian"`` uses the Box-Muller variant of the noise instead; ``out`` receives
    the result when given."""
    lib = load()
    if noise not in _NOISE:
        raise ValueError("noise must be 'uniform' or 'gaussian'")
    seeds = _seeds(seeds)
    fitness = _fitness(fitness, pop_size, seeds)
    dev = _device(fitness, seeds)
    g = _out(out, (int(n_params),), dev)
    with torch.cuda.device(dev):
        st = lib.vn_gradient_ex(_ptr(fitness), _ptr(seeds), pop_size, int(n_params), float(sigma),
                                int(offset) & _M64, _NOISE[noise], _ptr(g), _stream(g))
    check(st, "vn_gradient_ex")
    return g


def gradient_update(fitness: torch.Tensor, seeds: torch.Tensor, theta: torch.Tensor, sigma: float,
                    pop_size: int, lr: float, offset: int = 0, *, noise: str = "uniform",
                    out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """The flat gradient estimate and the ES step in one launch (``vn_gradient_update``):
    grad = virtual_flat_gradient(fitness, seeds, theta.numel(), sigma, pop_size, offset),
    then theta += lr * grad in place (fp32 fma). Returns grad (in ``out`` when given); both
    are bit-identical to the two separate calls."""
    lib = load()
    if noise not in _NOISE:
        raise ValueError("noise must be 'uniform' or 'gaussian'")
    if not isinstance(theta, torch.Tensor) or not theta.is_cuda or not theta.is_contiguous() \
            or theta.dtype != torch.float32:
        raise ValueError("theta must be a contiguous float32 CUDA tensor (updated in place)")
    seeds = _seeds(seeds)
    fitness = _fitness(fitness, pop_size, seeds)
    dev = _device(fitness, seeds, theta)
    g = _out(out, (theta.numel(),), dev)
    with torch.cuda.device(dev):
        st = lib.vn_gradient_update(_ptr(fitness), _ptr(seeds), pop_size, theta.numel(), float(sigma),
                                    int(offset) & _M64, _NOISE[noise], float(lr), _ptr(g), _ptr(theta),
                                    _stream(g))
    check(st, "vn_gradient_update")
    return g


def noise_dump(seeds: torch.Tensor, n_elements: int, offset: int, *,
               noise: str = "uniform", out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """(pop, n) fp32 noise, D[i, t] = PRNG(seed_i, offset + t): the centered uniform
    (bit-exact), or with ``noise="gaussian"`` the Box-Muller variant; written into ``out``
    when given."""
    lib = load()
    if noise not in _NOISE:
        raise ValueError("noise must be 'uniform' or 'gaussian'")
    seeds = _seeds(seeds)
    d = _out(out, (seeds.numel(), int(n_elements)), seeds.device)
    with torch.cuda.device(seeds.device):
        st = lib.vn_noise_dump_ex(_ptr(seeds), seeds.numel(), int(n_elements), int(offset) & _M64,
                                  _NOISE[noise], _ptr(d), _stream(d))
    check(st, "vn_noise_dump")
    return d


def virtual_reduce_metric(center: torch.Tensor, seeds: torch.Tensor, sigma: float, n_params: int,
                          offset: int = 0, *, out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """fitness[i] = mean_k |center[k] + sigma * noise[i, k]|, (pop,) fp32 (in ``out`` when given)."""
    lib = load()
    center = _cuda(center, "center").reshape(-1).to(torch.float32)
    if center.numel() != n_params:
        raise ValueError(f"center has {center.numel()} elements, n_params={n_params}")
    seeds = _seeds(seeds)
    dev = _device(center, seeds)
    f = _out(out, (seeds.numel(),), dev)
    with torch.cuda.device(dev):
        st = lib.vn_reduce_metric(_ptr(center), _ptr(seeds), seeds.numel(), int(n_params),
                                  float(sigma), int(offset) & _M64, _ptr(f), _stream(f))
    check(st, "vn_reduce_metric")
    return f


def centered_ranks(fitness: torch.Tensor, *, out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Fitness shaping: rank (ascending, ties by index) / (pop - 1) - 0.5, float32 (pop,)."""
    lib = load()
    fitness = _cuda(fitness, "fitness").reshape(-1).to(torch.float32)
    pop = fitness.numel()
    if out is None:
        out = torch.empty(pop, dtype=torch.float32, device=fitness.device)
    elif out.shape != (pop,) or out.dtype != torch.float32 or not out.is_contiguous():
        raise ValueError("out must be a contiguous float32 tensor of shape (pop,)")
    with torch.cuda.device(_device(fitness, out)):
        st = lib.vn_centered_ranks(_ptr(fitness), pop, _ptr(out), _stream(fitness))
    check(st, "vn_centered_ranks")
    return out


def es_update(theta: torch.Tensor, grad: torch.Tensor, lr: float) -> torch.Tensor:
    """theta += lr * grad in place (float32, contiguous, same number of elements); returns theta."""
    lib = load()
    if not isinstance(theta, torch.Tensor) or not theta.is_cuda or not theta.is_contiguous() \
            or theta.dtype != torch.float32:
        raise ValueError("theta must be a contiguous float32 CUDA tensor (updated in place)")
    grad = _cuda(grad, "grad").to(torch.float32)
    if grad.numel() != theta.numel():
        raise ValueError("grad and theta differ in size")
    with torch.cuda.device(_device(theta, grad)):
        st = lib.vn_es_update(_ptr(theta), _ptr(grad), theta.numel(), float(lr), _stream(theta))
    check(st, "vn_es_update")
    return theta


def hash_probe(seed: int, offset: int, n_sums: int, m: int, *, device=None,
               out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """The hash alone (``vn_hash_probe``, a measurement kernel): (n_sums,) fp32 with
    sums[t] = sum_{e < m} PRNG(seed, offset + t*m + e)."""
    lib = load()
    dev = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
    s = _out(out, (int(n_sums),), dev)
    with torch.cuda.device(dev):
        st = lib.vn_hash_probe(int(seed), int(offset) & _M64, int(n_sums), int(m), _ptr(s), _stream(s))
    check(st, "vn_hash_probe")
    return s


def compute_offsets(param_shapes: Sequence[Sequence[int]]) -> list:
    """Start offset of each parameter block: the element count of all blocks before it."""
    offsets, total = [], 0
    for shape in param_shapes:
        offsets.append(total)
        total += math.prod(int(d) for d in shape)
    return offsets


def perturbed_linear_path(x: torch.Tensor, weight: torch.Tensor) -> str:
    """"tc" or "ffma": the kernel ``virtual_perturbed_linear`` would use (no launch)."""
    lib = load()
    for t, name in ((x, "x"), (weight, "weight")):
        if not isinstance(t, torch.Tensor) or not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor")
    batch = x.shape[-2]
    with torch.cuda.device(_device(x, weight)):
        p = lib.vn_perturbed_linear_path(_ptr(x), _dt(x, "x"), int(x.dim() == 2), _ptr(weight),
                                         _dt(weight, "weight"), batch, weight.shape[1],
                                         weight.shape[0])
    return "tc" if p == _lib.VN_PATH_TC else "ffma"


def device_status(device=None) -> None:
    """Synchronise the current stream and raise VNError if a kernel recorded an expired wait
    since the last call (the status word is then cleared). Results written by the
    tensor-core forward since the last call are valid only if this returns normally."""
    lib = load()
    s = torch.cuda.current_stream(device)
    check(lib.vn_device_status(ctypes.c_void_p(s.cuda_stream)), "vn_device_status")


__all__ = ["virtual_perturbed_linear", "virtual_weight_gradient", "virtual_bias_gradient",
           "virtual_flat_gradient",
           "noise_dump", "virtual_reduce_metric", "compute_offsets", "perturbed_linear_path", "hash_probe",
           "device_status", "VNError"]
