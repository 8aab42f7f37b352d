"""The pins have teeth: plausible mistakes planted in copies of the oracle
(on the CPU, in a temporary directory) must each fail at least one pin."""
import os
import subprocess

import pytest

import oracle
from oracle_pins import ALL_PINS

SRC = os.path.join(os.path.dirname(oracle.__file__), "attn_oracle.c")

# (name, text in the definition, replacement) -- each a plausible slip.
MUTANTS = [
    ("scale_dropped", "srow[j] = dot * scale;", "srow[j] = dot;"),
    ("k_transposed", "dot += q[c] * kj[c];", "dot += q[c] * K[(c % sk) * d + (j % d)];"),
    ("causal_offset_sign", "int64_t diag = i + (sk - sq);", "int64_t diag = i - (sk - sq);"),
    ("causal_strict", "int64_t n = last + 1;", "int64_t n = last;"),
    ("lse_without_max", "*lse = m + log(l);", "*lse = log(l);"),
    ("not_normalised", "for (int64_t j = 0; j < n; ++j) srow[j] /= l;", ""),
    ("v_dims_reversed", "o[c] += p * vj[c];", "o[c] += p * vj[d - 1 - c];"),
    ("exp_base_2", "srow[j] = exp(srow[j] - m);", "srow[j] = exp2(srow[j] - m);"),
    ("max_not_subtracted_twice", "srow[j] = exp(srow[j] - m);", "srow[j] = exp(srow[j] - 2 * m);"),
    ("online_prev_not_rescaled", "double l_new = a_prev * l_prev + a_cur * row_l;",
     "double l_new = l_prev + a_cur * row_l;"),
    ("online_o_not_rescaled", "oi[c] = (l_prev * a_prev * oi[c] + a_cur * pv[c]) / l_new;",
     "oi[c] = (l_prev * oi[c] + a_cur * pv[c]) / l_new;"),
    ("online_tile_overlap", "for (int64_t j0 = 0; j0 < sk; j0 += bc) {",
     "for (int64_t j0 = 0; j0 < sk; j0 += (bc > 1 ? bc - 1 : 1)) {"),
    ("head_stride_wrong", "const double *Kh = k + head * sk * d;\n                const double *Vh = v + head * sk * d;\n                double l_out;",
     "const double *Kh = k; /* head offset forgotten */\n                const double *Vh = v + head * sk * d;\n                double l_out;"),
    # backward
    ("bwd_D_dropped", "dP[i * sk + j] = P[i * sk + j] * (dP[i * sk + j] - Di);",
     "dP[i * sk + j] = P[i * sk + j] * dP[i * sk + j];"),
    ("bwd_dk_scale_dropped", "dK[j * d + c] = scale * ak;", "dK[j * d + c] = ak;"),
    ("bwd_dv_uses_ds", "av += P[i * sk + j] * dO[i * d + c];", "av += dP[i * sk + j] * dO[i * d + c];"),
    ("bwd_dq_uses_v", "acc += dP[i * sk + j] * K[j * d + c];", "acc += dP[i * sk + j] * V[j * d + c];"),
    ("bwd_dp_indices_swapped", "for (int64_t c = 0; c < d; ++c) acc += dO[i * d + c] * V[j * d + c];",
     "for (int64_t c = 0; c < d; ++c) acc += dO[(j % sq) * d + c] * V[(i % sk) * d + c];"),
    ("bwd_rows_D_dropped", "acc += prow[j] * (dprow[j] - Di) * k_head[j * d + c];",
     "acc += prow[j] * dprow[j] * k_head[j * d + c];"),
    ("bwd_cols_scale_dropped", "dKj[c] += scale * ds * qi[c];", "dKj[c] += ds * qi[c];"),
    ("bwd_cols_mask_ignored", "if (j > last_visible_key(i, sq, sk, causal)) continue;", ""),
    # KV cache
    ("kv_append_at_zero", "int64_t pos = start + t;", "int64_t pos = t;"),
    ("kv_new_not_attended", "int64_t valid = clamp_len(cache_len[e], s_cache) + s_new;",
     "int64_t valid = clamp_len(cache_len[e], s_cache);"),
    ("kv_batch_index_wrong", "int64_t e = plane / h;", "int64_t e = plane % b;"),
    ("kv_write_stops_early", "if (pos >= s_cache) break; /* no room left in the cache */",
     "if (pos >= s_cache - 1) break;"),
    ("bwd_probs_strict_mask", "int64_t n = 1 + last; /* visible keys 0..last */",
     "int64_t n = last; /* visible keys 0..last-1 */"),
]


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(tmp_path, name, old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site for {name} not unique/present"
    path = tmp_path / f"{name}.c"
    path.write_text(src.replace(old, new))
    so = tmp_path / f"lib{name}.so"
    subprocess.run(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-fopenmp", str(path),
                    "-o", str(so), "-lm"], check=True)
    lib = oracle.load_library(str(so))
    caught = []
    for pin in ALL_PINS:
        if pin(lib):
            caught.append(pin.__name__)
    assert caught, f"no pin caught mutant {name}"
