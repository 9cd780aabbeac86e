"""Plant a mistake in a copy of the oracle and check that some pin catches it.

Each mutant is the oracle source with one plausible error: a dropped term,
a wrong sign or index, a transposed operand, an off-by-one, a wrong tie
order.  Every mutation stays inside the buffers it touches, so a mutant can
only return wrong numbers, never corrupt memory.  The pins must reject
every mutant.
"""

import os

import pytest

import oracle
import pins

MUTANTS = {
    "relu dropped": ("double relu = dot > 0.0 ? dot : 0.0;", "double relu = dot;"),
    "nibble order swapped": ("(d % 2 == 0) ? (byte & 0x0F) : (byte >> 4)",
                             "(d % 2 == 0) ? (byte >> 4) : (byte & 0x0F)"),
    "scale group index": ("scales[d / 32]", "scales[(d / 32 + 1) % 4]"),
    "e4m3 exponent bias": ("v = ldexp(1.0 + (double)m / 8.0, e - 7);",
                           "v = ldexp(1.0 + (double)m / 8.0, e - 8);"),
    "e4m3 subnormal": ("v = ldexp((double)m / 8.0, -6);", "v = ldexp((double)m / 8.0, -7);"),
    "e2m1 mantissa": ("v = ldexp(1.0 + (double)m / 2.0, e - 1);",
                      "v = ldexp(1.0 + (double)m / 4.0, e - 1);"),
    "e2m1 sign": ("int sign = (nibble >> 3) & 1;", "int sign = (nibble >> 2) & 1;"),
    "ue8m0 bias": ("return ldexp(1.0, (int)code - 127);", "return ldexp(1.0, (int)code - 128);"),
    "bf16 half": ("uint32_t u = (uint32_t)bits << 16;", "uint32_t u = (uint32_t)bits << 15;"),
    "q scale dropped": ("q[i] = smq_oracle_e4m3(q8[i]) * (double)q_scale;",
                        "q[i] = smq_oracle_e4m3(q8[i]);"),
    "head weight dropped": ("logit += w[h] * relu;", "logit += relu;"),
    "weight sign": ("logit += w[h] * relu;", "logit += fabs(w[h]) * relu;"),
    "q transposed": ("dot += q[h * D + d] * k[d];", "dot += q[(d % H) * D + (h + d) % D] * k[d];"),
    "page walk skipped": ("int64_t page = bt_row[slot];\n  if (page < 0 || page >= num_pages) return -1;\n  const uint8_t *base = k_cache + page * page_bytes;\n  const uint8_t *vals",
                          "int64_t page = slot % num_pages;\n  if (page < 0 || page >= num_pages) return -1;\n  const uint8_t *base = k_cache + page * page_bytes;\n  const uint8_t *vals"),
    "token offset": ("const uint8_t *vals = base + tok * (D / 2);",
                     "const uint8_t *vals = base + ((tok + 1) % page_size) * (D / 2);"),
    "contig ks ignored": ("int64_t row = ks + p;", "int64_t row = p;"),
    "mask block offset": ("int64_t p = b * cbs + j;", "int64_t p = b * cbs + j + 1;"),
    "mask accepts -1": ("if (b < 0) continue;", "if (b < -1) continue;\n    if (b < 0) b = 0;"),
    "top-k ascending": ("if (x->v > y->v) return -1;\n  if (x->v < y->v) return 1;",
                        "if (x->v > y->v) return 1;\n  if (x->v < y->v) return -1;"),
    "tie order": ("return (x->p > y->p) - (x->p < y->p);", "return (x->p < y->p) - (x->p > y->p);"),
    "no -1 pad": ("out[j] = (j < n) ? (int32_t)s[j].p : -1;", "out[j] = (j < n) ? (int32_t)s[j].p : 0;"),
    "expansion keeps repeats": ("if (nu == 0 || kept[nu - 1] != kept[i]) kept[nu++] = kept[i];",
                                "kept[nu++] = kept[i];"),
    "expansion end rounds up": ("cols += (L - start < sbkv) ? (L - start) : sbkv;", "cols += sbkv;"),
    "encode ties to odd": ("if (dc < db || (dc == db && (c % 2) == 0)) best = c;",
                           "if (dc < db || (dc == db && (c % 2) == 1)) best = c;"),
    "encode without saturation": ("if (a > table[n - 1]) a = table[n - 1]; /* saturation */", "/* no saturation */"),
    "k scale against 4": ("while (6.0 * ldexp(1.0, e) < amax) ++e;", "while (4.0 * ldexp(1.0, e) < amax) ++e;"),
    "k scale clamp": ("if (code < 1) code = 1;", "if (code < 0) code = 0;"),
    "k nibbles swapped": ("values[(32 * g + i) / 2] = (uint8_t)(lo | (hi << 4));",
                          "values[(32 * g + i) / 2] = (uint8_t)(hi | (lo << 4));"),
    "k slot offset": ("int64_t page = s / page_size, off = s % page_size;",
                      "int64_t page = s / page_size, off = (s + 1) % page_size;"),
    "k scales placement": ("base + (int64_t)page_size * (D / 2) + off * (D / 32)) != 0)",
                           "base + (int64_t)page_size * (D / 2) + (off ^ 1) * (D / 32)) != 0)"),
    "q scale 447": ("float s = amax > 0.0f ? amax / 448.0f : 1.0f;", "float s = amax > 0.0f ? amax / 447.0f : 1.0f;"),
    "q zero-row scale": ("float s = amax > 0.0f ? amax / 448.0f : 1.0f;", "float s = amax > 0.0f ? amax / 448.0f : 0.5f;"),
    "bf16 ties down": ("if (dhi < dlo || (dhi == dlo && (hi & 1) == 0)) return hi;", "if (dhi < dlo) return hi;"),
    "source ties to the higher id": ("return (x->b > y->b) - (x->b < y->b);", "return (x->b < y->b) - (x->b > y->b);"),
    "source block sum": ("if (logits[p] > m) m = logits[p];", "m = (m == -INFINITY ? 0.0 : m) + logits[p];"),
    "source partial block dropped": ("int64_t nb = L > 0 ? (L + cbs - 1) / cbs : 0;", "int64_t nb = L > 0 ? L / cbs : 0;"),
    "source no -1 pad": ("cand[i] = i < nb ? (int32_t)s[i].b : -1;", "cand[i] = i < nb ? (int32_t)s[i].b : 0;"),
    "gather scale offset": ("base + (int64_t)page_size * (D / 2) + tok * (D / 32),\n           (size_t)(D / 32));",
                            "base + (int64_t)page_size * (D / 2),\n           (size_t)(D / 32));"),
}


def _caught(orc):
    for pin in pins.ALL_PINS:
        try:
            pin(orc)
        except (AssertionError, ValueError):
            return pin.__name__
    return None


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    with open(oracle.SOURCE) as f:
        src = f.read()
    assert src.count(old) == 1, f"mutation site for {name!r} not found exactly once"
    path = tmp_path / "mutant.c"
    path.write_text(src.replace(old, new))
    lib = oracle.build(str(tmp_path / "libmutant.so"), source=str(path))
    orc = oracle.Oracle(lib)
    caught_by = _caught(orc)
    assert caught_by is not None, f"no pin rejects the mutant {name!r}"


def test_unmutated_oracle_passes_every_pin():
    assert _caught(oracle.Oracle(oracle.build(os.path.join(os.path.dirname(oracle.DEFAULT_LIB),
                                                            "libsmq_oracle_check.so")))) is None
