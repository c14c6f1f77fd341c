"""Device-side fill of the seeded inputs (bit-identical to ``gen.InputSpec``)
through ``libkvqgen.so``; torch supplies the device buffers and the stream."""

from __future__ import annotations

import ctypes
import os

import numpy as np
import torch

from .gen import NORMAL_TABLE, TAU_TABLE, InputSpec

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB = None


def _lib():
    global _LIB
    if _LIB is None:
        path = os.path.join(_HERE, "libkvqgen.so")
        if not os.path.exists(path):
            raise ImportError(f"{path} is missing: run __graft_entry__.build() first")
        lib = ctypes.CDLL(path)
        vp, i, ll = ctypes.c_void_p, ctypes.c_int, ctypes.c_longlong
        lib.kvq_gen_kv.argtypes = [vp, vp, vp, vp, vp, vp, i, i, i, ll, ll, i, i, vp, vp, vp]
        lib.kvq_gen_kv.restype = i
        lib.kvq_gen_q.argtypes = [vp, vp, i, i, ll, i, vp, vp]
        lib.kvq_gen_q.restype = i
        _LIB = lib
    return _LIB


def _u64_tensor(values, device) -> torch.Tensor:
    arr = np.array([int(v) for v in values], dtype=np.uint64).view(np.int64)
    return torch.from_numpy(arr).to(device)


class DeviceInputs:
    """Fills device tensors with the synthetic K/V/q of ``spec``."""

    def __init__(self, spec: InputSpec, device="cuda"):
        self.spec = spec
        self.device = torch.device(device)
        self.normal = torch.from_numpy(NORMAL_TABLE).to(self.device)
        self.tau = torch.from_numpy(TAU_TABLE).to(self.device)
        self._sigma = {}
        self.dtype = torch.bfloat16 if spec.bf16 else torch.float32

    def sigma(self, layer: int) -> torch.Tensor:
        if layer not in self._sigma:
            self._sigma[layer] = torch.from_numpy(self.spec.sigma(layer)).to(self.device)
        return self._sigma[layer]

    def kv_block(self, layer: int, seq_begin: int, nseq: int, t0: int, n: int, out_k=None, out_v=None):
        s = self.spec
        H, D = s.n_kv_heads, s.head_dim
        shape = (nseq, H, n, D)
        if out_k is None:
            out_k = torch.empty(shape, dtype=self.dtype, device=self.device)
        if out_v is None:
            out_v = torch.empty(shape, dtype=self.dtype, device=self.device)
        assert tuple(out_k.shape) == shape and out_k.is_contiguous() and out_k.dtype == self.dtype
        assert tuple(out_v.shape) == shape and out_v.is_contiguous() and out_v.dtype == self.dtype
        units = [(b, h) for b in range(seq_begin, seq_begin + nseq) for h in range(H)]
        kk = _u64_tensor([s.key("K", layer, b, h) for b, h in units], self.device)
        vk = _u64_tensor([s.key("V", layer, b, h) for b, h in units], self.device)
        tk = _u64_tensor([s.key("tau", layer, b, h) for b, h in units], self.device)
        stream = torch.cuda.current_stream(self.device).cuda_stream
        rc = _lib().kvq_gen_kv(kk.data_ptr(), vk.data_ptr(), tk.data_ptr(), self.sigma(layer).data_ptr(),
                               self.normal.data_ptr(), self.tau.data_ptr(), len(units), H, D, t0, n,
                               int(s.bf16), int(s.spikes), out_k.data_ptr(), out_v.data_ptr(), stream)
        if rc != 0:
            raise RuntimeError(f"kvq_gen_kv failed ({rc})")
        # keep the key buffers alive until the fill has run
        torch.cuda.current_stream(self.device).synchronize()
        return out_k, out_v

    def q_block(self, layer: int, seq_begin: int, nseq: int, step: int, out=None):
        s = self.spec
        shape = (nseq, s.n_q_heads, s.head_dim)
        if out is None:
            out = torch.empty(shape, dtype=self.dtype, device=self.device)
        assert tuple(out.shape) == shape and out.is_contiguous() and out.dtype == self.dtype
        keys = _u64_tensor([s.key("q", layer, b, h) for b in range(seq_begin, seq_begin + nseq)
                            for h in range(s.n_q_heads)], self.device)
        stream = torch.cuda.current_stream(self.device).cuda_stream
        rc = _lib().kvq_gen_q(keys.data_ptr(), self.normal.data_ptr(), nseq * s.n_q_heads, s.head_dim,
                              step, int(s.bf16), out.data_ptr(), stream)
        if rc != 0:
            raise RuntimeError(f"kvq_gen_q failed ({rc})")
        torch.cuda.current_stream(self.device).synchronize()
        return out
