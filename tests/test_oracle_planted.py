"""Planted mistakes: each plausible error, planted in a private copy of the
oracle source and compiled on the CPU, must make at least one pin fail.
This shows the pins constrain every step of the oracle, not only its
happy path."""
import os
import subprocess

import pytest

import oracle
from tests import pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "ds4oracle.c")

# (name, exact source text, replacement)
PLANTS = [
    ("swap_scale_min", "    int sc = sb[g] & 15, mn = sb[g] >> 4;\n    int32_t dot = 0;\n    for (int i = 0; i < 16; i++) {\n      int e = 16 * g + i; /* element index within the superblock */\n      int q = (sb[16 + (e >> 2)]",
     "    int sc = sb[g] >> 4, mn = sb[g] & 15;\n    int32_t dot = 0;\n    for (int i = 0; i < 16; i++) {\n      int e = 16 * g + i; /* element index within the superblock */\n      int q = (sb[16 + (e >> 2)]"),
    ("min_term_sign", "rd16(sb + 82));\n      float m = dmin * (float)B;\n      float p = dx[b] * fmaf(d, (float)A, -m);",
     "rd16(sb + 82));\n      float m = dmin * (float)B;\n      float p = dx[b] * fmaf(d, (float)A, m);"),
    ("q4s_min_term_sign", "rd16(sb + 146));\n      float m = dmin * (float)B;\n      float p = dx[b] * fmaf(d, (float)A, -m);",
     "rd16(sb + 146));\n      float m = dmin * (float)B;\n      float p = dx[b] * fmaf(d, (float)A, m);"),
    ("q_bit_order", "int q = (sb[16 + (e >> 2)] >> (2 * (e & 3))) & 3;",
     "int q = (sb[16 + (e >> 2)] >> (6 - 2 * (e & 3))) & 3;"),
    ("round_half_even", "float r = roundf(x[i] / d);", "float r = rintf(x[i] / d);"),
    ("scale_128", "float d = amax / 127.0f;", "float d = amax / 128.0f;"),
    ("tie_to_higher", "if (best < 0 || key[e] > key[best]) best = e;",
     "if (best < 0 || key[e] >= key[best]) best = e;"),
    ("weights_from_keys", "w[j] = (s[ids[j]] / sum) * L->route_scale;",
     "w[j] = (key[ids[j]] / sum) * L->route_scale;"),
    ("exp_drop_term", "  p = fmaf(p, r, CAS_C2);\n", ""),
    ("silu_sign", "float ora_silu(float g) { return g / (1.0f + ora_exp(-g)); }",
     "float ora_silu(float g) { return g / (1.0f + ora_exp(g)); }"),
    ("swiglu_swapped", "h[j] = ora_silu(gj) * uj;", "h[j] = ora_silu(uj) * gj;"),
    ("drop_shared", "if (L->n_shared) acc = acc + c->a[((size_t)t * ns + k) * H + r];", ""),
    ("q8_offset", "s += (int32_t)(int8_t)blk[2 + i] * (int32_t)xq[i];",
     "s += (int32_t)(int8_t)blk[1 + i] * (int32_t)xq[i];"),
    ("q2s_block_index", "ora_q2s_dot(sb, b % 8, xq + 32 * b, gs + 2 * b, &A, &B);",
     "ora_q2s_dot(sb, b % 8, xq + 32 * (b % 8), gs + 2 * (b % 8), &A, &B);"),
    ("group_sum_8", "for (int i = 0; i < 16; i++) s += q[32 * b + 16 * g + i];",
     "for (int i = 0; i < 8; i++) s += q[32 * b + 16 * g + i];"),
    ("half_bias", "v = ldexpf((float)(man | 1024u), (int)ex - 25);", "v = ldexpf((float)(man | 1024u), (int)ex - 24);"),
    ("hash_weight", "float wk = 1.0f / (float)k;", "float wk = 1.0f / (float)(k + 1);"),
    ("rms_no_eps", "float inv = 1.0f / sqrtf(ss / (float)H + eps);", "float inv = 1.0f / sqrtf(ss / (float)H);"),
    ("no_route_scale", "w[j] = (s[ids[j]] / sum) * L->route_scale;", "w[j] = (s[ids[j]] / sum);"),
    ("down_uses_x", "expert_down_rows(L, e, c->hq + ts * F, c->dh + ts * (F / 32), c->gsh + ts * (F / 16), ch * CHUNK,",
     "expert_down_rows(L, e, c->xq + (size_t)t * H, c->dh + ts * (F / 32), c->gsh + ts * (F / 16), ch * CHUNK,"),
    ("bias_ignored", "key[e] = s[e] + L->router_bias[e];", "key[e] = s[e];"),
    ("expert_one_segment", "return units < 8 ? units : 8;", "return 1;"),
    ("expert_four_segments", "return units < 8 ? units : 8;", "return units < 4 ? units : 4;"),
    ("q4s_nibble_order", "int q = (sb[16 + (e >> 1)] >> (4 * (e & 1))) & 15;",
     "int q = (sb[16 + (e >> 1)] >> (4 - 4 * (e & 1))) & 15;"),
    ("q4s_scale_min_swap", "    int g = 2 * j + h;\n    int sc = sb[g] & 15, mn = sb[g] >> 4;\n    int32_t dot = 0;\n    for (int i = 0; i < 16; i++) {\n      int e = 16 * g + i; /* element index within the superblock */\n      int q = (sb[16 + (e >> 1)]",
     "    int g = 2 * j + h;\n    int sc = sb[g] >> 4, mn = sb[g] & 15;\n    int32_t dot = 0;\n    for (int i = 0; i < 16; i++) {\n      int e = 16 * g + i; /* element index within the superblock */\n      int q = (sb[16 + (e >> 1)]"),
    ("q4s_scale_offset", "float d = ora_half(rd16(sb + 144)), dmin = ora_half(rd16(sb + 146));",
     "float d = ora_half(rd16(sb + 146)), dmin = ora_half(rd16(sb + 144));"),
    ("dense_one_segment", "const int S = expert_segs(FMT_Q8_0, c->K);", "const int S = 1;"),
    ("dense_token_stride", "c->xq + (size_t)t * c->K,\n", "c->xq,\n"),
    ("dense_transposed", "c->y[(size_t)t * c->N + n] = ora_row(", "c->y[(size_t)n * c->T + t] = ora_row("),
    ("segments_merged", "    tot = tot + acc;\n  }\n  return tot;\n}\n\nstatic float row_q2s",
     "    tot = acc;\n  }\n  return tot;\n}\n\nstatic float row_q2s"),
]


@pytest.mark.parametrize("name,old,new", PLANTS, ids=[p[0] for p in PLANTS])
def test_planted_mistake_is_caught(tmp_path, name, old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, f"plant site for {name} not found exactly once"
    bad_src = tmp_path / "ds4oracle_planted.c"
    bad_src.write_text(src.replace(old, new))
    lib = tmp_path / "libplanted.so"
    subprocess.check_call(["gcc", *oracle.CFLAGS, "-o", str(lib), str(bad_src), "-lm"])
    bad = oracle.Oracle(str(lib))
    failed = []
    for check in pins.ALL_CHECKS:
        try:
            check(bad)
        except AssertionError:
            failed.append(check.__name__)
            break
    assert failed, f"planted mistake {name!r} passed every pin"
