"""Torch-facing convenience wrapper over the C ABI.

PyTorch supplies device memory and streams only; every step of insert and query
runs in libsbf's kernels.
"""
from __future__ import annotations

import numpy as np
import torch

from . import _native as N


def _stream_handle(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream)


def _check_device_u8(seq: torch.Tensor) -> None:
    if not (seq.is_cuda and seq.dtype == torch.uint8 and seq.is_contiguous()):
        raise ValueError("seq must be a contiguous uint8 CUDA tensor")


def _check_device_i64(off: torch.Tensor) -> None:
    if not (off.is_cuda and off.dtype == torch.int64 and off.is_contiguous() and off.dim() == 1):
        raise ValueError("offsets must be a contiguous 1-D int64 CUDA tensor")


class SuperBloomFilter:
    """An SBF on the current CUDA device (sbf_create / sbf_destroy)."""

    def __init__(self, num_bits: int, k: int = 31, m: int = 16, s: int = 28, H: int = 4,
                 seed: int = 0, alphabet="dna", sectors: str = "fixed", runtime_kernels: bool = False):
        """alphabet: "dna" (default), "protein" or "dna_triplet" (Sec. IV-A;
        k <= 32, 12, 10 respectively), or the SBF_ALPHABET_* value.
        sectors: "fixed" (the paper's layout, hash i in word i mod 4) or
        "hashed" (hash-chosen words for H < 4; SBF_FLAG_HASHED_SECTORS).
        runtime_kernels: always the runtime-parameter kernels
        (SBF_FLAG_RUNTIME_KERNELS)."""
        if sectors not in ("fixed", "hashed"):
            raise ValueError(f"sectors must be 'fixed' or 'hashed', not {sectors!r}")
        self.alphabet = N.alphabet_id(alphabet)
        self.sectors = sectors
        flags = (N.FLAG_HASHED_SECTORS if sectors == "hashed" else 0) | \
            (N.FLAG_RUNTIME_KERNELS if runtime_kernels else 0)
        self._h = N.sbf_create_ex(int(num_bits), k, m, s, H, seed, self.alphabet, flags)
        self.k, self.m, self.s, self.H = k, m, s, H
        self.seed = seed & (2**64 - 1)
        self.num_shards = N.sbf_num_shards(self._h)
        self.device = torch.cuda.current_device()

    @property
    def handle(self) -> int:
        return self._h

    @property
    def nbytes(self) -> int:
        return self.num_shards * 32

    @property
    def specialized(self) -> bool:
        return N.sbf_is_specialized(self._h)

    def close(self) -> None:
        if getattr(self, "_h", None):
            N.sbf_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    # ---- device-resident (stream-ordered, no synchronisation) -------------
    def insert(self, seq: torch.Tensor, offsets: torch.Tensor, stream=None) -> None:
        _check_device_u8(seq)
        _check_device_i64(offsets)
        N.sbf_insert(self._h, seq.data_ptr(), offsets.data_ptr(), offsets.numel() - 1,
                     _stream_handle(stream))

    def query(self, seq: torch.Tensor, offsets: torch.Tensor, out: torch.Tensor | None = None,
              stream=None, total_len: int | None = None) -> torch.Tensor:
        """Returns (or fills) an int32 tensor of answer words; bit g of word
        g >> 5 answers the k-mer at absolute position g.  Without `out` the
        length of the buffer is taken from total_len, else from seq."""
        _check_device_u8(seq)
        _check_device_i64(offsets)
        if out is None:
            n_pos = seq.numel() if total_len is None else total_len
            out = torch.zeros((n_pos + 31) // 32 + 1, dtype=torch.int32, device=seq.device)
        N.sbf_query(self._h, seq.data_ptr(), offsets.data_ptr(), offsets.numel() - 1,
                    out.data_ptr(), _stream_handle(stream))
        return out

    def query_dense(self, seq: torch.Tensor, record_len: int, out: torch.Tensor | None = None,
                    stream=None) -> torch.Tensor:
        """Query a dense batch of fixed-length records (seq.numel() //
        record_len of them); same answer layout as query()."""
        _check_device_u8(seq)
        n = seq.numel() // record_len
        if out is None:
            out = torch.zeros((n * record_len + 31) // 32 + 1, dtype=torch.int32, device=seq.device)
        N.sbf_query_dense(self._h, seq.data_ptr(), n, record_len, out.data_ptr(), _stream_handle(stream))
        return out

    # ---- host-resident (synchronising) ------------------------------------
    def insert_host(self, seq: np.ndarray, offsets: np.ndarray) -> None:
        seq = np.ascontiguousarray(seq, dtype=np.uint8)
        offsets = np.ascontiguousarray(offsets, dtype=np.int64)
        N.sbf_insert_host(self._h, seq.ctypes.data, offsets.ctypes.data, offsets.size - 1, 0)

    def query_host(self, seq: np.ndarray, offsets: np.ndarray, out: np.ndarray | None = None) -> np.ndarray:
        seq = np.ascontiguousarray(seq, dtype=np.uint8)
        offsets = np.ascontiguousarray(offsets, dtype=np.int64)
        if out is None:
            out = np.zeros((int(offsets[-1]) + 31) // 32 + 1, dtype=np.uint32)
        N.sbf_query_host(self._h, seq.ctypes.data, offsets.ctypes.data, offsets.size - 1,
                         out.ctypes.data, 0)
        return out

    # ---- image --------------------------------------------------------------
    def to_numpy(self) -> np.ndarray:
        """The raw image as uint64[num_shards, 4] (synchronises)."""
        host = np.empty((self.num_shards, 4), dtype=np.uint64)
        torch.cuda.current_stream().synchronize()
        N.sbf_copy_bits(self._h, host.ctypes.data, host.nbytes, 0)
        torch.cuda.synchronize()
        return host

    def to_tensor(self, stream=None) -> torch.Tensor:
        """The raw image as a device int64 tensor [num_shards, 4] (async copy)."""
        t = torch.empty((self.num_shards, 4), dtype=torch.int64, device=f"cuda:{self.device}")
        N.sbf_copy_bits(self._h, t.data_ptr(), self.nbytes, _stream_handle(stream))
        return t

    def load(self, image) -> None:
        if isinstance(image, torch.Tensor):
            N.sbf_load_bits(self._h, image.data_ptr(), image.numel() * image.element_size(),
                            _stream_handle(None))
        else:
            image = np.ascontiguousarray(image, dtype=np.uint64)
            N.sbf_load_bits(self._h, image.ctypes.data, image.nbytes, 0)
            torch.cuda.synchronize()

    def clear(self, stream=None) -> None:
        N.sbf_clear(self._h, _stream_handle(stream))

    def status(self, stream=None) -> int:
        return N.sbf_get_status(self._h, _stream_handle(stream))
