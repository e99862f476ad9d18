"""Plant one plausible mistake at a time in a copy of the oracle (on the CPU) and
check that at least one pin catches it.  This shows the pins are strong enough
to catch a dropped term, a wrong sign, a wrong index or a transposed operand."""

import os
import tempfile

import pytest

import oracle
import oracle_pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "q2k_oracle.c")

# (name, text in the oracle source, replacement)
MUTANTS = [
    ("f16_bias", "(int)expo - 25", "(int)expo - 24"),
    ("f16_subnormal_scale", "ldexp((double)frac, -24)", "ldexp((double)frac, -25)"),
    ("nibbles_swapped", "const float dl = d * (float)(sc & 0x0F);",
     "const float dl = d * (float)(sc >> 4);"),
    ("min_uses_dl_nibble", "const float ml = dmin * (float)(sc >> 4);",
     "const float ml = dmin * (float)(sc & 0x0F);"),
    ("min_sign", "out[pushed++] = prod - ml;", "out[pushed++] = prod + ml;"),
    ("min_dropped", "out[pushed++] = prod - ml;", "out[pushed++] = prod;"),
    ("d_dmin_swapped", "const float d = q2ko_f16_to_f32(load_le16(block + 80));",
     "const float d = q2ko_f16_to_f32(load_le16(block + 82));"),
    ("q_offset_transposed", "const int q_offset = half * 32 + segment * 16;",
     "const int q_offset = half * 16 + segment * 32;"),
    ("q_mask_3bits", "& 0x03;", "& 0x07;"),
    ("loop_order_segment_outer",
     "for (int shift = 0; shift <= 6; shift += 2) {\n            for (int segment = 0; segment < 2; ++segment) {",
     "for (int segment = 0; segment < 2; ++segment) {\n            for (int shift = 0; shift <= 6; shift += 2) {"),
    ("fma_like_fused", "const float prod = dl * (float)q;\n                    out[pushed++] = prod - ml;",
     "out[pushed++] = (float)((double)dl * (double)q - (double)ml * 1.0000001);"),
    ("big_endian_d", "return (uint16_t)(p[0] | (p[1] << 8));", "return (uint16_t)(p[1] | (p[0] << 8));"),
    ("x_transposed", "const float *xrow = job->x + m * job->K;", "const float *xrow = job->x + m;"),
    ("y_transposed", "job->y[m * job->N + n] = acc;", "job->y[n * job->M + m] = acc;"),
    ("last_block_dropped", "for (size_t b = 0; b < blocks_per_row; ++b)\n            q2ko_dequant_block(wrow",
     "for (size_t b = 0; b + 1 < blocks_per_row; ++b)\n            q2ko_dequant_block(wrow"),
    ("abs_dropped", "acc_abs += fabs(term);", "acc_abs += term;"),
    ("dequant_allows_short_out", "if (n_out != n_blocks * ORACLE_QK_K)", "if (n_out < n_blocks * ORACLE_QK_K - 1)"),
]


@pytest.fixture(scope="module")
def src_text():
    with open(SRC) as f:
        return f.read()


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(tmp_path, src_text, name, old, new):
    assert src_text.count(old) >= 1, f"mutation site for {name} not found"
    mutated = src_text.replace(old, new, 1)
    src = tmp_path / f"mut_{name}.c"
    src.write_text(mutated)
    lib = oracle.build(force=True, src=str(src), out=str(tmp_path / f"lib_{name}.so"))
    o = oracle.Oracle(lib)
    caught = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(o)
        except (AssertionError, oracle.OracleError):
            caught.append(pin.__name__)
    assert caught, f"no pin caught mutant {name}"


# Mistakes in the Python compositions (batched and routed products), planted by
# overriding one helper of a copy of the oracle object.
class _SlotAsToken(oracle.Oracle):
    def route_token(self, route, top_k):
        return route % top_k


class _PackedExperts(oracle.Oracle):
    def expert_bytes(self, w, expert, n, K, expert_stride):
        return super().expert_bytes(w, expert, n, K, n * (K // 256) * 84)


class _SlottedUsesToken(oracle.Oracle):
    def matmul_id(self, x, w, ids, n, n_experts, expert_stride, top_k, threads=1, slotted=False):
        if slotted:  # the mistake: read the token's row as the unslotted product does
            x = x[::top_k].copy()
            slotted = False
        return super().matmul_id(x, w, ids, n, n_experts, expert_stride, top_k, threads, slotted)


class _BatchesSwapped(oracle.Oracle):
    def matmul_batched_mv(self, x, w, n, threads=1):
        return super().matmul_batched_mv(x[::-1].copy(), w, n, threads)


@pytest.mark.parametrize("cls", [_SlotAsToken, _PackedExperts, _BatchesSwapped, _SlottedUsesToken],
                         ids=lambda c: c.__name__)
def test_composition_mutant_is_caught(cls):
    o = cls(oracle.default().path)
    caught = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(o)
        except (AssertionError, oracle.OracleError):
            caught.append(pin.__name__)
    assert caught, f"no pin caught {cls.__name__}"
