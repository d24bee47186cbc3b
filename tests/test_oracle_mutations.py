"""Planted mistakes in the oracle must be caught by its pins (CPU only).

Each case copies ``oracle/pkv_oracle.cpp``, plants one plausible mistake (a
wrong index, a dropped term, a flipped sign, a transposed operand, an
off-by-one), compiles the copy into a temporary library and runs every pin
against it. At least one pin has to fail, otherwise the pins would not have
noticed that mistake in the real oracle either.
"""

import os
import subprocess
import sys

import pytest


SOURCE = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle",
                      "pkv_oracle.cpp")

# (name, original text, planted text, which occurrence of the original)
MUTATIONS = [
    ("logical page uses t mod P", "int logical = t / g->page_size;",
     "int logical = t % g->page_size;", 0),
    ("slot uses t div P", "int slot = t % g->page_size;", "int slot = t / g->page_size;", 0),
    ("pool layout [page][slot][kv][d]",
     "return ((static_cast<size_t>(page) * g->num_kv_heads + kv_head) * g->page_size + slot) *",
     "return ((static_cast<size_t>(page) * g->page_size + slot) * g->num_kv_heads + kv_head) *",
     0),
    ("scale 1/D instead of 1/sqrt(D)", "const double scale = 1.0 / std::sqrt(static_cast<double>(D));",
     "const double scale = 1.0 / static_cast<double>(D);", 0),
    ("score sign flipped", "s[t] = dot * scale;", "s[t] = -dot * scale;", 0),
    ("max kept in the numerator", "double w = std::exp(s[t] - m) / z;",
     "double w = std::exp(s[t]) / z;", 0),
    ("weights normalised by count", "double w = std::exp(s[t] - m) / z;",
     "double w = std::exp(s[t] - m) / len;", 0),
    ("values weighted from K", "out[d] += w * v_rows[", "out[d] += w * k_rows[", 0),
    ("GQA heads interleaved", "size_t row = static_cast<size_t>(b) * g->num_q_heads + h;",
     "size_t row = static_cast<size_t>(b) * g->num_q_heads + (h % group) * g->num_kv_heads + kv;",
     0),
    ("appended token not attended", "const int len = seq_lens[b];",
     "const int len = seq_lens[b] - 1;", 0),
    ("append slot off by one", "int slot = pos % g->page_size;",
     "int slot = (pos + 1) % g->page_size;", 0),
    ("append writes V into K", "k_pool[pool_index(g, page, kv, slot, d)] = k_new[src];",
     "k_pool[pool_index(g, page, kv, slot, d)] = v_new[src];", 0),
    ("merge drops the rescale of l", "if (l[s] > 0.0) denom += std::exp(m[s] - big) * l[s];",
     "if (l[s] > 0.0) denom += l[s];", 0),
    ("split range drops its last token", "if (t1 > len) t1 = len;",
     "if (t1 > len) t1 = len - 1;", 0),
    ("split scale dropped", "const double scale = 1.0 / std::sqrt(static_cast<double>(D));",
     "const double scale = 1.0;", 1),
    ("contiguous cache read transposed",
     "size_t src = (static_cast<size_t>(t) * num_kv_heads + kv) * D + d;",
     "size_t src = (static_cast<size_t>(kv) * len + t) * D + d;", 0),
    ("threaded variant skips sequences", "for (int b = w; b < batch; b += nthreads)",
     "for (int b = w + 1; b < batch; b += nthreads)", 0),
    ("prefill token does not attend itself", "start_pos[b] + i + 1, D,", "start_pos[b] + i, D,",
     0),
    ("prefill fill ignores the chunk start",
     "const int pos = start_pos[b] + (row - cu_tokens[b]);",
     "const int pos = row - cu_tokens[b];", 0),
    ("prefill reads the next sequence's queries",
     "const size_t row = static_cast<size_t>(cu_tokens[b] + i);",
     "const size_t row = static_cast<size_t>(cu_tokens[b] + i + (b + 1 < batch ? 1 : 0));", 0),
    ("prefill gathers one key too few", "const int len = start_pos[b] + n;          // keys",
     "const int len = start_pos[b] + n - 1;      // keys", 0),
    ("key rotation sign flipped", "rotated[row + i] = float_to_bf16_rne(xc - ys);",
     "rotated[row + i] = float_to_bf16_rne(xc + ys);", 0),
    ("key rotation pairs neighbours", "const float y = bf16_bits_to_float(k_new[row + i + half]);",
     "const float y = bf16_bits_to_float(k_new[row + (i ^ 1)]);", 0),
    ("key rotation uses the next position's cosine",
     "const float c = cos_t[static_cast<size_t>(pos) * half + i];",
     "const float c = cos_t[static_cast<size_t>(pos + 1) * half + i];", 0),
    ("key rotation uses the previous position's sine",
     "const float s = sin_t[static_cast<size_t>(pos) * half + i];",
     "const float s = sin_t[static_cast<size_t>(pos - 1) * half + i];", 0),
    ("key rotation reads the sequence index's row",
     "const float c = cos_t[static_cast<size_t>(pos) * half + i];",
     "const float c = cos_t[static_cast<size_t>(b) * half + i];", 0),
    ("key rotation drops the sine term", "rotated[row + i + half] = float_to_bf16_rne(yc + xs);",
     "rotated[row + i + half] = float_to_bf16_rne(yc);", 0),
    ("query rotation swaps cos and sin", "q_out[row + i + half] = y * c + x * s;",
     "q_out[row + i + half] = y * s + x * c;", 0),
    ("query rotation uses the wrong position",
     "const double c = cos_t[static_cast<size_t>(pos) * half + i];",
     "const double c = cos_t[static_cast<size_t>(pos + 1) * half + i];", 0),
]


def _plant(text, old, new, nth):
    at = -1
    for _ in range(nth + 1):
        at = text.find(old, at + 1)
        assert at >= 0, f"snippet not found: {old}"
    return text[:at] + new + text[at + len(old):]


def _pins_failed_by(tmp_path, text):
    """Names of the pins a build of `text` fails, or None if it crashed."""
    mutant_src = tmp_path / "mutant.cpp"
    mutant_src.write_text(text)
    lib = tmp_path / "libmutant.so"
    subprocess.run(["g++", "-std=c++17", "-O1", "-ffp-contract=off", "-fPIC", "-shared",
                    "-pthread", "-o", str(lib),
                    str(mutant_src)], check=True)
    # run the pins in a child process: a planted index mistake may read out
    # of bounds, and a crash counts as noticed too
    code = (
        "import sys, oracle, oracle_pins\n"
        "print('READY', flush=True)\n"
        f"m = oracle.Oracle({str(lib)!r})\n"
        "bad = []\n"
        "for pin in oracle_pins.ALL_PINS:\n"
        "    try:\n"
        "        pin(m)\n"
        "    except AssertionError:\n"
        "        bad.append(pin.__name__)\n"
        "print('CAUGHT', ' '.join(bad))\n"
    )
    here = os.path.dirname(os.path.abspath(__file__))
    env = dict(os.environ, PYTHONPATH=os.pathsep.join([here, os.path.dirname(here)]))
    run = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env,
                         timeout=600)
    assert "READY" in run.stdout, run.stderr[-2000:]
    if run.returncode != 0:
        return None  # the build crashed or raised inside a pin
    line = [x for x in run.stdout.splitlines() if x.startswith("CAUGHT")][-1]
    return line.split()[1:]


def test_unmodified_oracle_passes_every_pin(tmp_path):
    with open(SOURCE) as f:
        assert _pins_failed_by(tmp_path, f.read()) == []


@pytest.mark.parametrize("name,old,new,nth", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_is_caught(tmp_path, name, old, new, nth):
    with open(SOURCE) as f:
        text = f.read()
    failed = _pins_failed_by(tmp_path, _plant(text, old, new, nth))
    assert failed is None or failed, f"no pin noticed: {name}"
