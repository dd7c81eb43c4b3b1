"""Seeded synthetic inputs shared by the CUDA path's tests/bench and the oracle.

Nothing here computes any step of the outer synchronisation: the module only
describes workload shapes and fills host arrays with reproducible random
numbers (see ``gen.c`` for the generator's published definitions).

Workloads (shapes and distributions follow the five configurations of the
outer-step benchmark; sizes are computed from the model dimensions):

* ``worked_example`` - one 4096x4096 fp32 tensor, K=3 learners, the tensor of
  the INTELLECT-1 notes' worked example (section 3.2): theta_g ~ N(0, 0.02),
  theta_k = theta_g - N(0, 1.2e-3).
* ``decoder_1b`` - a 1.1B decoder-shaped tensor set (22 layers, d=2048,
  FFN 5632, 32 q / 4 kv heads, vocab 32000, untied embedding), K=4, per-tensor
  Delta ~ N(0, sigma_t) with sigma_t log-uniform in [3e-4, 3e-3].
* ``decoder_10b`` - a 10B decoder-shaped set (42 layers, d=4096, FFN 14336,
  32 q / 8 kv heads, vocab 128256), K=14, Delta ~ N(0, 1.2e-3), several
  outer steps.
* ``ragged_heavy`` - 2000 tensors with sizes log-uniform in [64, 16Mi]
  (every 10th forced to 4096), K=8, Delta = 1e-3 * Student-t(3).
* ``quorum_10b`` - the 10B shapes, K=16 learners, a seeded random present
  subset of size 1..16 and weights ~ U[0.5, 1.5] per (fragment, outer step).
* ``learner_1b`` / ``learner_10b`` - one learner (K=1) quantising its whole
  1.1B / 10B model for transmission: every tensor in one ragged batch, no
  merge (the INTELLECT-1 notes' worked example, section 3.2 steps 4-5, at
  full-model scale).
"""
from __future__ import annotations

import ctypes
import math
import os
from dataclasses import dataclass, field

import numpy as np

from ._build import load_library

SEED = 0xD110C0

# stream kinds (first label of a stream key)
_K_THETA = 1
_K_REPLICA = 2
_K_TENSOR_PARAM = 3
_K_SIZES = 4
_K_QUORUM = 5
_K_WEIGHTS = 6
_K_MOMENTUM = 7

_lib = None


def lib():
    global _lib
    if _lib is None:
        L = load_library()
        u64, i64, i32, f64 = ctypes.c_uint64, ctypes.c_int64, ctypes.c_int32, ctypes.c_double
        vp = ctypes.c_void_p
        L.synth_key.restype = u64
        L.synth_key.argtypes = [u64, u64, u64, u64]
        L.synth_words.restype = None
        L.synth_words.argtypes = [u64, i64, i64, vp]
        L.synth_uniform.restype = None
        L.synth_uniform.argtypes = [u64, i64, i64, vp]
        L.synth_normal_f32.restype = None
        L.synth_normal_f32.argtypes = [u64, i64, i64, f64, f64, vp]
        L.synth_replica_f32.restype = None
        L.synth_replica_f32.argtypes = [u64, i64, i64, vp, f64, i32, vp]
        _lib = L
    return _lib


def key(seed: int, kind: int, step: int, a: int, b: int) -> int:
    return int(lib().synth_key(seed & (2**64 - 1), (kind << 32) | step, a, b))


def words(k: int, start: int, n: int) -> np.ndarray:
    out = np.empty(n, dtype=np.uint64)
    lib().synth_words(k, start, n, out.ctypes.data)
    return out


def uniform(k: int, start: int, n: int) -> np.ndarray:
    out = np.empty(n, dtype=np.float64)
    lib().synth_uniform(k, start, n, out.ctypes.data)
    return out


def normal_f32(k: int, start: int, n: int, mean: float, std: float, out=None) -> np.ndarray:
    if out is None:
        out = np.empty(n, dtype=np.float32)
    assert out.dtype == np.float32 and out.flags.c_contiguous and out.size == n
    lib().synth_normal_f32(k, start, n, mean, std, out.ctypes.data)
    return out


def replica_f32(k: int, start: int, base: np.ndarray, scale: float, dist: int, out=None):
    base = np.ascontiguousarray(base, dtype=np.float32)
    n = base.size
    if out is None:
        out = np.empty(n, dtype=np.float32)
    assert out.dtype == np.float32 and out.flags.c_contiguous and out.size == n
    lib().synth_replica_f32(k, start, n, base.ctypes.data, scale, dist, out.ctypes.data)
    return out


# ----------------------------------------------------------------------------
# model shapes


def decoder_tensor_numels(layers, d, ffn, n_q, n_kv, vocab):
    """numel of every tensor of a decoder, in model order: embedding, per layer
    (q, k, v, o, gate, up, down, two RMSNorm vectors), final norm, lm_head."""
    head = d // n_q
    kv = n_kv * head
    out = [vocab * d]
    for _ in range(layers):
        out += [d * d, d * kv, d * kv, d * d, ffn * d, ffn * d, d * ffn, d, d]
    out += [d, vocab * d]
    return out


def decoder_1b_numels():
    return decoder_tensor_numels(22, 2048, 5632, 32, 4, 32000)


def decoder_10b_numels():
    return decoder_tensor_numels(42, 4096, 14336, 32, 8, 128256)


def ragged_heavy_numels(n_tensors=2000, seed=SEED + 4):
    u = uniform(key(seed, _K_SIZES, 0, 0, 0), 0, n_tensors)
    lo, hi = math.log(64.0), math.log(16 * 1024 * 1024)
    sizes = np.floor(np.exp(lo + (hi - lo) * u)).astype(np.int64)
    sizes = np.clip(sizes, 64, 16 * 1024 * 1024)
    sizes[9::10] = 4096  # every 10th tensor is a norm vector
    return [int(s) for s in sizes]


# ----------------------------------------------------------------------------
# workloads


@dataclass
class Workload:
    name: str
    numels: list
    K: int
    seed: int
    delta_dist: int = 0            # 0 normal, 1 Student-t(3)
    delta_scale: float = 1.2e-3    # scale of Delta (or per-tensor, see below)
    per_tensor_sigma: bool = False  # sigma_t log-uniform in [3e-4, 3e-3]
    theta_std: float = 0.02
    n_frags: int = 1
    steps: int = 1
    quorum: bool = False            # random present subsets and weights
    role: str = "syncer"            # "learner": stats + quantise only, K=1
    description: str = ""
    _sigmas: list = field(default=None, repr=False)

    @property
    def n_tensors(self):
        return len(self.numels)

    @property
    def n_elems(self):
        return int(sum(self.numels))

    def tensor_scale(self, t: int) -> float:
        if not self.per_tensor_sigma:
            return self.delta_scale
        if self._sigmas is None:
            u = uniform(key(self.seed, _K_TENSOR_PARAM, 0, 0, 0), 0, self.n_tensors)
            lo, hi = math.log(3e-4), math.log(3e-3)
            self._sigmas = [float(math.exp(lo + (hi - lo) * x)) for x in u]
        return self._sigmas[t]

    def theta_global(self, t: int, out=None, n=None) -> np.ndarray:
        """Initial global parameters of tensor t (its first n values if n is
        given: the generator is counter-based, so a prefix is the same values)."""
        return normal_f32(key(self.seed, _K_THETA, 0, t, 0), 0,
                          self.numels[t] if n is None else n, 0.0, self.theta_std, out)

    def replica(self, k: int, t: int, base: np.ndarray, step: int = 0, out=None):
        """Learner k's copy of tensor t after its inner steps: base - scale * X."""
        return replica_f32(key(self.seed, _K_REPLICA, step, t, k), 0, base,
                           self.tensor_scale(t), self.delta_dist, out)

    def momentum(self, t: int, out=None) -> np.ndarray:
        """A non-zero momentum state for tests that start mid-run."""
        return normal_f32(key(self.seed, _K_MOMENTUM, 0, t, 0), 0, self.numels[t], 0.0,
                          1e-3, out)

    def present(self, frag: int, step: int) -> np.ndarray:
        """Present mask (uint8[K]) of one merge; all present unless quorum."""
        if not self.quorum:
            return np.ones(self.K, dtype=np.uint8)
        u = uniform(key(self.seed, _K_QUORUM, step, frag, 0), 0, self.K + 1)
        size = 1 + min(int(u[0] * self.K), self.K - 1)
        order = np.argsort(u[1:], kind="stable")
        mask = np.zeros(self.K, dtype=np.uint8)
        mask[order[:size]] = 1
        return mask

    def weights(self, frag: int, step: int) -> np.ndarray:
        """Merge weights (float32[K]): all 1, or tokens-processed ~ U[0.5, 1.5]."""
        if not self.quorum:
            return np.ones(self.K, dtype=np.float32)
        u = uniform(key(self.seed, _K_WEIGHTS, step, frag, 0), 0, self.K)
        return (0.5 + u).astype(np.float32)


def worked_example(K=3):
    return Workload("worked_example", [4096 * 4096], K, SEED + 1,
                    description="one 4096x4096 fp32 tensor, K=3, all weights 1")


def decoder_1b(K=4):
    return Workload("decoder_1b", decoder_1b_numels(), K, SEED + 2, per_tensor_sigma=True,
                    n_frags=24,
                    description="1.1B decoder set (201 tensors), K=4, P=24 fragments")


def decoder_10b(K=14, steps=3):
    return Workload("decoder_10b", decoder_10b_numels(), K, SEED + 3, n_frags=24,
                    steps=steps,
                    description="10B decoder set (381 tensors), K=14, P=24, 3 outer steps")


def ragged_heavy(K=8, n_tensors=2000):
    return Workload("ragged_heavy", ragged_heavy_numels(n_tensors), K, SEED + 4,
                    delta_dist=1, delta_scale=1e-3,
                    description="2000 ragged tensors 64..16Mi, K=8, Delta=1e-3*t3")


def quorum_10b(K=16, steps=4):
    return Workload("quorum_10b", decoder_10b_numels(), K, SEED + 5, n_frags=24,
                    steps=steps, quorum=True,
                    description="10B shapes, K=16, random quorum 1..16, weights U[0.5,1.5]")


def learner_1b():
    return Workload("learner_1b", decoder_1b_numels(), 1, SEED + 6, per_tensor_sigma=True,
                    role="learner",
                    description="one learner quantises its whole 1.1B decoder set "
                                "(201 tensors) as one ragged batch, K=1")


def learner_10b():
    return Workload("learner_10b", decoder_10b_numels(), 1, SEED + 7, role="learner",
                    description="one learner quantises its whole 10B decoder set "
                                "(381 tensors) as one ragged batch, K=1")


WORKLOADS = {
    "worked_example": worked_example,
    "decoder_1b": decoder_1b,
    "decoder_10b": decoder_10b,
    "ragged_heavy": ragged_heavy,
    "quorum_10b": quorum_10b,
    "learner_1b": learner_1b,
    "learner_10b": learner_10b,
}


def offsets_of(numels) -> np.ndarray:
    off = np.zeros(len(numels) + 1, dtype=np.int64)
    np.cumsum(np.asarray(numels, dtype=np.int64), out=off[1:])
    return off


def n_threads() -> int:
    return int(os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1))
