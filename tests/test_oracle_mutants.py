"""The oracle's pins must catch plausible mistakes.

Each mutant below is a one-line mistake planted in a copy of the oracle's C
source (on the CPU, in a temporary directory): a wrong divisor, a sum in
place of a maximum, a transposed head index, a reversed tie-break, a missing
cap, and so on.  The whole pin suite of test_oracle_pins.py is rerun against
each mutant build; at least one pin must fail for every mutant.
"""
import inspect
import os
import subprocess
import tempfile

import pytest

import oracle
import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "oasis_oracle.c")

MUTANTS = {
    "summary divides by bs-1": ("(float)(sum / (double)bs)", "(float)(sum / (double)(bs - 1))"),
    "summary skips last token": ("for (int t = 0; t < bs; ++t) {\n                        size_t idx",
                                 "for (int t = 0; t < bs - 1; ++t) {\n                        size_t idx"),
    "score takes the minimum": ("if (dot > best) best = dot;", "if (dot < best || best == -INFINITY) best = dot;"),
    "score sums over drafts": ("if (dot > best) best = dot;", "best = (best == -INFINITY ? 0.0 : best) + dot;"),
    "score GQA index transposed": ("(((size_t)b * L + l) * Hq + (size_t)h * G + g) * D",
                                   "(((size_t)b * L + l) * Hq + (size_t)g * H + h) * D"),
    "score draft/batch index swapped": ("(((size_t)b * L + l) * Hq + (size_t)h * G + g) * D",
                                        "(((size_t)l * B + b) * Hq + (size_t)h * G + g) * D"),
    "min/max summary rows swapped": ("summ_mm[(blk * 2 + 0) * D + d] = hi;", "summ_mm[(blk * 2 + 0) * D + d] = lo;"),
    "min/max summary skips token 0": ("uint16_t hi = k[(blk * bs) * D + d], lo = hi;",
                                      "uint16_t hi = k[(blk * bs + 1) * D + d], lo = hi;"),
    "min/max score takes the lower product": ("bound += lo > hi ? lo : hi;", "bound += lo < hi ? lo : hi;"),
    "min/max score sums over drafts": ("if (bound > best) best = bound;",
                                       "best = (best == -INFINITY ? 0.0 : best) + bound;"),
    "ctx top-K window at the end of the capacity": (
        "const int win_begin = n - c->local_blocks > 0 ? n - c->local_blocks : 0;",
        "const int win_begin = NB - c->local_blocks > 0 ? NB - c->local_blocks : 0;"),
    "ctx top-K keeps scores past the context": ("rest[nr].s = j < n ? sc[j] : -INFINITY;", "rest[nr].s = sc[j];"),
    "append summary divides by bs": ("(float)(sum / (double)(t + 1))", "(float)(sum / (double)bs)"),
    "append evicts the most recent": ("lu[q] < lu[best] || (lu[q] == lu[best]", "lu[q] > lu[best] || (lu[q] == lu[best]"),
    "append skips the earlier rows": ("for (int r = 0; r < t; ++r) {", "for (int r = 0; r < 0; ++r) {"),
    "append keeps the context length": ("ctx_len[b] = p + 1;", "ctx_len[b] = p;"),
    "top-k ties to higher id": ("    return (a->id > b->id) - (a->id < b->id);\n}\n\n/*\n * Per-KV-head",
                                "    return (a->id < b->id) - (a->id > b->id);\n}\n\n/*\n * Per-KV-head"),
    "top-k sorts ascending": ("if (a->s > b->s) return -1;\n    if (a->s < b->s) return 1;",
                              "if (a->s < b->s) return -1;\n    if (a->s > b->s) return 1;"),
    "local window off by one": ("j >= c->num_blocks - c->local_blocks", "j > c->num_blocks - c->local_blocks"),
    "cap ignored": ("n = nm < cap ? nm : cap;", "n = nm;"),
    "cap floors": ("cap = (int)ceil(r * (double)slots_of(c) - 1e-6);", "cap = (int)floor(r * (double)slots_of(c));"),
    "LRU evicts most recent": ("if (a->last != b->last) return (a->last > b->last) - (a->last < b->last);",
                               "if (a->last != b->last) return (a->last < b->last) - (a->last > b->last);"),
    "hits not marked used": ("                    lu[s] = step;\n                    in_p[s] = 1;",
                             "                    in_p[s] = 1;"),
    "fetched blocks keep priority order": ("qsort(fetched, (size_t)n, sizeof(int32_t), cmp_int32);", ""),
    "fetch copies K into V": ("memcpy(pool_v + (u * S + s) * blk_elems, host_v", "memcpy(pool_v + (u * S + s) * blk_elems, host_k"),
    "attention drops the scale": ("double w = exp(x * scale - mx);", "double w = exp(x - mx);"),
    "attention mask off by one": ("(int64_t)j * bs + t >= ctx_len[b]", "(int64_t)j * bs + t > ctx_len[b]", "all"),
    "attention GQA index transposed": ("const int hq = h * G + g;", "const int hq = g * H + h;"),
    "attention skips the normalisation": ("o[d] = den > 0.0 ? (float)(acc[d] / den) : 0.0f;",
                                          "o[d] = den > 0.0 ? (float)(acc[d]) : 0.0f;"),
    "plan evicts one block too many": ("e = nres + n - S;", "e = nres + n - S + 1;"),
    "plan evicts though slots are empty": ("e = nres + n - S;", "e = n;"),
    "fetched blocks not marked used": ("                sob[fetched[r]] = s;\n                lu[s] = step;",
                                       "                sob[fetched[r]] = s;"),
    "free slots taken from the top": ("for (int s = 0; s < S; ++s) {\n                int free_slot",
                                      "for (int s = S - 1; s >= 0; --s) {\n                int free_slot"),
    "refresh reads the whole block": ("for (int r = 0; r <= t; ++r) {\n                    sum +=",
                                      "for (int r = 0; r < bs; ++r) {\n                    sum +="),
}


def _pin_functions():
    return [f for name, f in inspect.getmembers(pins, inspect.isfunction)
            if name.startswith("test_") and not inspect.signature(f).parameters]


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name):
    old, new, *mode = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation site not found for {name!r}"
    mutated = src.replace(old, new) if mode == ["all"] else src.replace(old, new, 1)
    with tempfile.TemporaryDirectory() as td:
        c_path = os.path.join(td, "oasis_oracle.c")
        with open(c_path, "w") as f:
            f.write(mutated)
        hdr = os.path.join(os.path.dirname(SRC), "oasis_oracle.h")
        so = os.path.join(td, "libmutant.so")
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-I", os.path.dirname(hdr),
                               "-o", so, c_path, "-lm"])
        caught = []
        with oracle.using_library(so):
            for f in _pin_functions():
                try:
                    f()
                except Exception:  # an assertion or a rejected call: the pin noticed
                    caught.append(f.__name__)
        assert caught, f"no pin catches the mutant {name!r}"
