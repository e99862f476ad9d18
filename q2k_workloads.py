"""Seeded synthetic inputs for the Q2_K matmul, dequantize and gather calls.

This module is shared by the oracle side (``oracle/``, the tests) and the CUDA
side (``bench.py``, the GPU tests).  It holds no arithmetic of the Q2_K method:
it only draws raw block bytes and activations, and restates the two input
fixtures that the mlx-native test page "tests/deepseek_q2_k.rs" builds
(``block(seed)`` and ``input(rows)``).

Block layout being generated (page "tests/deepseek_q2_k.rs", constants
``QK_K``/``BLOCK_BYTES`` and the ``block`` fixture): 84 bytes per 256 weights,
bytes 0..15 packed scale/min nibbles, bytes 16..79 the 2-bit quants, bytes
80..81 the f16 ``d`` and bytes 82..83 the f16 ``dmin``, both little endian.

Recipe for the seeded workloads (one ``numpy.random.default_rng(seed)`` per
workload, seed = the workload's index in ``WORKLOADS``), in this draw order:

1. all scale bytes, shape ``[n_blocks, 16]``, uniform over 0..255;
2. all quant bytes, shape ``[n_blocks, 64]``, uniform over 0..255;
3. ``d`` for every block: float64 uniform on [0.001, 0.05), rounded to
   binary16 (round to nearest even, ``astype(float16)``);
4. ``dmin`` for every block, drawn the same way;
5. the activations ``x``: ``standard_normal((M, K), dtype=float32)``;
6. gather ids, where the workload has them: ``integers(0, vocab, n_tokens)``.

Blocks are laid out row-major: block ``b`` of weight row ``n`` sits at byte
``(n * (K // 256) + b) * 84``.
"""

from __future__ import annotations

import dataclasses

import numpy as np

QK_K = 256
BLOCK_BYTES = 84
GGML_TYPE_Q2_K = 10


def random_blocks(rng: np.random.Generator, n_blocks: int) -> np.ndarray:
    """Draw ``n_blocks`` Q2_K blocks as a flat uint8 array of ``n_blocks*84`` bytes."""
    scales = rng.integers(0, 256, size=(n_blocks, 16), dtype=np.uint8)
    qs = rng.integers(0, 256, size=(n_blocks, 64), dtype=np.uint8)
    d = rng.uniform(0.001, 0.05, size=n_blocks).astype(np.float16)
    dmin = rng.uniform(0.001, 0.05, size=n_blocks).astype(np.float16)
    out = np.empty((n_blocks, BLOCK_BYTES), dtype=np.uint8)
    out[:, 0:16] = scales
    out[:, 16:80] = qs
    out[:, 80:82] = d.astype("<f2").view(np.uint8).reshape(n_blocks, 2)
    out[:, 82:84] = dmin.astype("<f2").view(np.uint8).reshape(n_blocks, 2)
    return out.reshape(-1)


def random_activations(rng: np.random.Generator, m: int, k: int) -> np.ndarray:
    return rng.standard_normal((m, k), dtype=np.float32)


# --- the page's own fixtures ("tests/deepseek_q2_k.rs", fns block and input) ---

def page_block(seed: int) -> np.ndarray:
    """The page's deterministic block fixture ``block(seed)`` as 84 uint8 bytes.

    Group g's byte holds scale ``(g + seed) % 15 + 1`` in the low nibble and
    min ``15 - ((3 g + seed) % 16)`` in the high nibble (u8 wrapping adds);
    quant byte i is ``73 i + 19 seed`` (mod 256); d = 0.125, dmin = 0.0625.
    """
    s = seed & 0xFF
    out = bytearray()
    for g in range(16):
        scale = ((g + s) & 0xFF) % 15 + 1
        mn = 15 - ((((g * 3) & 0xFF) + s) & 0xFF) % 16
        out.append(((mn << 4) | scale) & 0xFF)
    for i in range(64):
        out.append((i * 73 + s * 19) & 0xFF)
    out += np.array([0.125], dtype="<f2").tobytes()
    out += np.array([0.0625], dtype="<f2").tobytes()
    assert len(out) == BLOCK_BYTES
    return np.frombuffer(bytes(out), dtype=np.uint8).copy()


def page_input(rows: int) -> np.ndarray:
    """The page's activation fixture ``input(rows)``: ``((17 i + 11) % 97)/48 - 1``."""
    i = np.arange(rows * QK_K, dtype=np.int64)
    return (((i * 17 + 11) % 97).astype(np.float32) / np.float32(48.0)
            - np.float32(1.0)).reshape(rows, QK_K)


# --- the five seeded workloads ---

@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    seed: int
    m: int
    n: int
    k: int
    gather_vocab: int = 0
    gather_tokens: int = 0
    gather_ids: tuple = ()

    @property
    def blocks_per_row(self) -> int:
        return self.k // QK_K

    @property
    def weight_bytes(self) -> int:
        return self.n * self.blocks_per_row * BLOCK_BYTES

    @property
    def flops(self) -> int:
        return 2 * self.m * self.n * self.k


WORKLOADS = (
    Workload("tiny", 0, 4, 8, 256, gather_vocab=8, gather_tokens=2, gather_ids=(2, 0)),
    Workload("decode_gemv_4096", 1, 1, 4096, 4096),
    Workload("ffn_pair", 2, 1, 14336, 4096),  # the pair's second half is FFN_DOWN
    Workload("spec_verify_m16", 3, 16, 4096, 4096, gather_vocab=32000, gather_tokens=16),
    Workload("prefill_m512", 4, 512, 7168, 7168),
)
FFN_DOWN = Workload("ffn_pair_down", 2, 1, 4096, 14336)


@dataclasses.dataclass(frozen=True)
class RoutedWorkload:
    """An expert-routed (mm_id) product: n_tokens tokens, top_k experts each, from
    a pool of n_experts [n, k] matrices packed back to back."""
    name: str
    seed: int
    n_tokens: int
    top_k: int
    n: int
    k: int
    n_experts: int

    @property
    def expert_bytes(self) -> int:
        return self.n * (self.k // QK_K) * BLOCK_BYTES


# Decode step of a DeepSeek-style MoE layer: one token, 8 of 64 experts of hidden
# size 7168 and expert width 2048 (a 308 MB pool, larger than L2).
MOE_DECODE = RoutedWorkload("moe_decode_top8", 5, 1, 8, 2048, 7168, 64)
# Prefill of the same layer: 512 tokens, so about 64 routes per expert.
MOE_PREFILL = RoutedWorkload("moe_prefill_top8", 6, 512, 8, 2048, 7168, 64)
# Eight decode GEMVs of the 4096 x 4096 workload in one batched launch.
BATCHED_DECODE_BATCHES = 8


def make_routed_ids(wl: RoutedWorkload, draw: int) -> np.ndarray:
    """Token-major expert ids: each token's top_k distinct experts, drawn from
    seed (wl.seed, draw)."""
    rng = np.random.default_rng([wl.seed, draw])
    return np.concatenate([rng.choice(wl.n_experts, wl.top_k, replace=False)
                           for _ in range(wl.n_tokens)]).astype(np.uint32)


def by_name(name: str) -> Workload:
    for w in WORKLOADS + (FFN_DOWN,):
        if w.name == name:
            return w
    raise KeyError(name)


@dataclasses.dataclass
class MatmulInputs:
    x: np.ndarray        # float32 [m, k]
    w: np.ndarray        # uint8 [n * k/256 * 84]
    ids: np.ndarray | None = None     # uint32 [n_tokens]
    table: np.ndarray | None = None   # uint8 [vocab * k/256 * 84]


def make_inputs(wl: Workload, with_gather: bool = True) -> MatmulInputs:
    """Seeded inputs of one workload (see the module docstring for the recipe).

    The tiny workload's weights are its 8 random rows; its gather table is the
    same 8 rows (vocab 8 x dim 256) and its ids are the fixed ``[2, 0]``.  For
    the M=16 workload the gather table is a separate 32000 x 4096 table drawn
    after the activations.
    """
    rng = np.random.default_rng(wl.seed)
    w = random_blocks(rng, wl.n * wl.blocks_per_row)
    x = random_activations(rng, wl.m, wl.k)
    out = MatmulInputs(x=x, w=w)
    if with_gather and wl.gather_tokens:
        if wl.gather_ids:
            out.ids = np.array(wl.gather_ids, dtype=np.uint32)
            out.table = w
        else:
            out.table = random_blocks(rng, wl.gather_vocab * wl.blocks_per_row)
            out.ids = rng.integers(0, wl.gather_vocab, size=wl.gather_tokens).astype(np.uint32)
    return out


def make_matmul_inputs(seed: int, m: int, n: int, k: int):
    """Ad-hoc seeded (x, w) for parity cases of arbitrary shape (same recipe)."""
    rng = np.random.default_rng(seed)
    w = random_blocks(rng, n * (k // QK_K))
    x = random_activations(rng, m, k)
    return x, w
