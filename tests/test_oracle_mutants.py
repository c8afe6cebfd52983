"""Planted mistakes: every mutated copy of the oracle must fail at least one pin.

Each mutant replaces one snippet of oracle/pa_oracle.c (a dropped term, a wrong
index, an off-by-one, a wrong sign or a missing normalisation), is compiled
into a temporary library on the CPU, and is run against the pins.  If some pin
would let a plausible mistake through, this test fails.
"""
import pytest

import oracle
import oracle_pins as pins

MUTANTS = {
    "kv_head_modulo": ("h / g,\n                        q + (size_t)row * head_dim, scale, 0, seq_lens[b]",
                       "h % num_kv_heads,\n                        q + (size_t)row * head_dim, scale, 0, seq_lens[b]"),
    "scale_dropped": ("s[t - t_begin] = scale * dot;", "s[t - t_begin] = dot;"),
    "decode_drops_last_key": ("scale, 0, seq_lens[b], out + (size_t)row * head_dim",
                              "scale, 0, seq_lens[b] - 1, out + (size_t)row * head_dim"),
    "head_ignored_in_pool": ("((size_t)blk * pool->num_kv_heads + kvh) * pool->block_size + off",
                             "((size_t)blk * pool->num_kv_heads + 0) * pool->block_size + off"),
    "offset_from_block_index": ("int32_t off = t % pool->block_size;", "int32_t off = (t / pool->block_size) % pool->block_size;"),
    "lse_without_log_l": ("*lse = m + log(l);", "*lse = m;"),
    "combine_unnormalised": ("for (int32_t e = 0; e < head_dim; ++e) o[e] /= wsum;", ""),
    "causal_off_by_one": ("scale, 0, pos + 1,", "scale, 0, pos,"),
    "chunk_start_ignores_chunk": ("const int32_t pos = L - C + (tok - cu_q_lens[s]);",
                                  "const int32_t pos = L - 1 + (tok - cu_q_lens[s]);"),
    "append_head_order": ("size_t dst = (((size_t)blk * num_kv_heads + h) * block_size + off) * head_dim;",
                          "size_t dst = (((size_t)blk * block_size + off) * num_kv_heads + h) * head_dim;"),
    "softmax_sign": ("double w = exp(s[t - t_begin] - m);", "double w = exp(m - s[t - t_begin]);"),
    "partition_size_floor": ("const int32_t per = (nb + num_partitions - 1) / num_partitions;",
                             "const int32_t per = nb / num_partitions > 0 ? nb / num_partitions : 1;"),
    "q_row_of_kv_head": ("q + (size_t)row * head_dim, scale, 0, seq_lens[b]",
                         "q + ((size_t)b * num_heads + (h / g) * g) * head_dim, scale, 0, seq_lens[b]"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    before, after = MUTANTS[name]
    src = oracle.SOURCE.read_text()
    assert src.count(before) == 1, f"snippet for {name} not found exactly once"
    mutated = tmp_path / "pa_oracle_mutant.c"
    mutated.write_text(src.replace(before, after))
    lib = oracle.build(mutated, tmp_path / "libmutant.so", force=True)
    mut = oracle.Oracle(lib)
    failures = []
    for pin in pins.ALL_PINS:
        try:
            pin(mut)
        except AssertionError as e:
            failures.append(pin.__name__)
        except oracle.OracleError:
            failures.append(pin.__name__ + " (error)")
    assert failures, f"planted mistake {name!r} passed every pin"
