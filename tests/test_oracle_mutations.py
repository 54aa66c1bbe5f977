"""Plant plausible mistakes in copies of the oracle and check that the pins
catch each one (CPU only; the planted copies live in a temporary directory,
never in the source tree)."""
import os

import pytest

import oracle
import oracle_pins

# (name, text to find, replacement, which occurrence (0-based) or None = all)
MUTATIONS = [
    ("causal mask off by one", "return !causal || pos_k <= pos_q;", "return !causal || pos_k < pos_q;", None),
    ("scale 1/d instead of 1/sqrt(d)", "1.0 / sqrt((double)d)", "1.0 / (double)d", None),
    ("rescale sign flipped", "exp(ma - mm)", "exp(mm - ma)", None),
    ("merge drops the rescale of l_a", "*l = a * la + b * lb;", "*l = la + b * lb;", None),
    ("merge uses a for both sides of O", "o[c] = a * oa[c] + b * ob[c];", "o[c] = a * oa[c] + a * ob[c];", None),
    ("ring rotates the wrong way", "int j = (r - s) % P;", "int j = (r + s) % P;", None),
    ("striped positions swapped for contiguous",
     "if (layout == ORACLE_LAYOUT_STRIPED) return i * (long)P + r;",
     "if (layout == ORACLE_LAYOUT_STRIPED) return (long)r * n + i;", None),
    ("lse misses the log", "double l = m + log(sum);", "double l = m + sum;", None),
    ("finalize does not divide by l", "o[c] = ost[c] / l;", "o[c] = ost[c];", None),
    ("scores use V instead of K (dense)",
     "s[kk] = scale * dot_q_k(qrow, kb + (size_t)kk * d, d);",
     "s[kk] = scale * dot_q_k(qrow, vb + (size_t)kk * d, d);", 0),
    ("value rows reversed (dense)", "const uint16_t* vr = vb + (size_t)kk * d;",
     "const uint16_t* vr = vb + (size_t)(N - 1 - kk) * d;", 0),
    ("no max subtraction (dense)", "sum += exp(s[kk] - m);\n      double l = m + log(sum);",
     "sum += exp(s[kk]);\n      double l = log(sum);", None),
    ("block weight scaled by a constant", "double w = exp(s[kk] - m);\n      l += w;",
     "double w = 0.5 * exp(s[kk] - m);\n      l += w;", None),
    ("zigzag second chunk off by one",
     "return i < c ? (long)r * c + i : (long)(2 * P - 1 - r) * c + (i - c);",
     "return i < c ? (long)r * c + i : (long)(2 * P - 2 - r) * c + (i - c);", None),
    ("zigzag halves in the wrong order",
     "return i < c ? (long)r * c + i : (long)(2 * P - 1 - r) * c + (i - c);",
     "return i < c ? (long)(2 * P - 1 - r) * c + i : (long)r * c + (i - c);", None),
    ("sliding window off by one", "if (window > 0 && pos_q - pos_k >= window) return 0;",
     "if (window > 0 && pos_q - pos_k > window) return 0;", None),
    ("sliding window ignored", "if (window > 0 && pos_q - pos_k >= window) return 0;", "", None),
    ("block partial ignores the mask in the sum",
     "      if (!allowed(causal, window, seg, pos_q, kpos[kk])) continue;\n      double w",
     "      double w", None),
    ("backward dS drops the D term (dense)",
     "const double ds = p * (dot_q_k(dorow, vb + (size_t)kk * d, d) - Dt);",
     "const double ds = p * dot_q_k(dorow, vb + (size_t)kk * d, d);", 0),
    ("backward dK without the scale (dense)", "gk[c] += scale * ds * widen_bf16(qrow[c]);",
     "gk[c] += ds * widen_bf16(qrow[c]);", None),
    ("backward dV weighted by dS instead of P (dense)", "gv[c] += p * widen_bf16(dorow[c]);",
     "gv[c] += ds * widen_bf16(dorow[c]);", None),
    ("backward D taken as zero (dense)", "      D[idx] = Dt;", "      D[idx] = 0.0;", None),
    ("backward dQ against V instead of K (dense)",
     "for (int c = 0; c < d; ++c) g[c] += scale * ds * widen_bf16(kb[(size_t)kk * d + c]);",
     "for (int c = 0; c < d; ++c) g[c] += scale * ds * widen_bf16(vb[(size_t)kk * d + c]);", 0),
    ("ring backward passes accumulators the wrong way", "const int to = (r + 1) % P;",
     "const int to = (r + P - 1) % P;", None),
    ("ring backward drops D", "const double ds = p * (dot_q_k(dorow, vrow, d) - D[tq]);",
     "const double ds = p * dot_q_k(dorow, vrow, d);", None),
    ("ring backward dQ uses q instead of k", "g[c] += scale * ds * widen_bf16(krow[c]);",
     "g[c] += scale * ds * widen_bf16(qrow[c]);", None),
    ("ring backward ignores the saved lse",
     "const double p = exp(scale * dot_q_k(qrow, krow, d) - lse[base + tq]);",
     "const double p = exp(scale * dot_q_k(qrow, krow, d));", None),
    ("sampled backward dV uses the query's q",
     "gv[c] += p * widen_bf16(ob[(size_t)t * d + c]);", "gv[c] += p * widen_bf16(qb[(size_t)t * d + c]);", None),
    ("backward from saved statistics drops D",
     "const double ds = p * (dot_q_k(dorow, vrow, d) - Dt);", "const double ds = p * dot_q_k(dorow, vrow, d);", None),
    ("backward from saved statistics takes D from the wrong row",
     "const double* orow = out + ((size_t)bh * N + t) * d;", "const double* orow = out + ((size_t)bh * N + kk) * d;",
     None),
    ("segment rule ignored", "  if (seg && seg[pos_q] != seg[pos_k]) return 0;\n", "", None),
    ("segment rule compares the query with a neighbour",
     "  if (seg && seg[pos_q] != seg[pos_k]) return 0;",
     "  if (seg && pos_k > 0 && seg[pos_q] != seg[pos_k - 1]) return 0;", None),
]


def _mutate(src: str, old: str, new: str, which):
    count = src.count(old)
    assert count >= 1, f"mutation anchor not found: {old!r}"
    if which is None:
        return src.replace(old, new)
    idx = -1
    for _ in range(which + 1):
        idx = src.index(old, idx + 1)
    return src[:idx] + new + src[idx + len(old):]


@pytest.mark.parametrize("name,old,new,which", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_pins_catch_planted_mistake(tmp_path, name, old, new, which):
    src = open(oracle.SOURCE, encoding="utf-8").read()
    mutated = _mutate(src, old, new, which)
    assert mutated != src
    c_path = tmp_path / "mutant.c"
    c_path.write_text(mutated, encoding="utf-8")
    so_path = str(tmp_path / "libmutant.so")
    oracle.build(str(c_path), so_path, force=True)
    orc = oracle.Oracle(so_path)
    failures = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(orc)
        except AssertionError as e:
            failures.append(f"{pin.__name__}: {str(e)[:80]}")
    assert failures, f"no pin caught the planted mistake: {name}"
    print(f"{name}: caught by {len(failures)} pin(s): {failures[0]}")
    assert os.path.dirname(so_path) != os.path.dirname(oracle.LIBRARY)
