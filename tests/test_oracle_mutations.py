"""Plants plausible mistakes in a copy of the oracle and checks that the pins catch them.

Each mutation edits one expression of oracle.c (in a temporary copy, on the CPU),
builds it, and runs tests/test_oracle_pins.py against that build.  A mutation that
survives means the pins do not constrain that part of the oracle.
"""
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "oracle.c")

MUTATIONS = {
    "nibble_order_swapped": (
        "int q = (k % 2 == 0) ? (byte & 0xF) : ((byte >> 4) & 0xF);",
        "int q = (k % 2 == 1) ? (byte & 0xF) : ((byte >> 4) & 0xF);"),
    "offset_dropped": (
        "return (double)(q - 8) * scale;",
        "return (double)(q) * scale;"),
    "offset_sign": (
        "return (double)(q - 8) * scale;",
        "return (double)(8 - q) * scale;"),
    "scale_index_transposed": (
        "double scale = oracle_f16_to_double(s[g * N + n]);",
        "double scale = oracle_f16_to_double(s[n * (K / G) + g]);"),
    "group_of_k": (
        "int64_t g = k / G;",
        "int64_t g = k % (K / G);"),
    "e4m3_bias": (
        "v = ldexp((double)(8 + m), e - 10);        /* 1.m * 2^(e-7) */",
        "v = ldexp((double)(8 + m), e - 9);        /* 1.m * 2^(e-7) */"),
    "e4m3_subnormal": (
        "v = ldexp((double)m, -9);                  /* 0.m * 2^-6 */",
        "v = ldexp((double)m, -10);                  /* 0.m * 2^-6 */"),
    "e2m1_exponent": (
        "v = ldexp((double)(2 + m), e - 2);         /* 1.m * 2^(e-1) */",
        "v = ldexp((double)(2 + m), e - 1);         /* 1.m * 2^(e-1) */"),
    "fp4_block_stride": (
        "double sfv = oracle_e4m3_to_double(sf[n * (K / 16) + k / 16]);",
        "double sfv = oracle_e4m3_to_double(sf[n * (K / 16) + k / 32]);"),
    "fp4_nibble_order": (
        "uint8_t code = (k % 2 == 0) ? (byte & 0xF) : ((byte >> 4) & 0xF);",
        "uint8_t code = (k % 2 == 0) ? ((byte >> 4) & 0xF) : (byte & 0xF);"),
    "fp8_alpha_dropped": (
        "out[i * ncols + j] = alpha * acc + b;",
        "out[i * ncols + j] = acc + b;"),
    "fp4_alpha_dropped": (
        "out[i * ncols + j] = alpha * acc;",
        "out[i * ncols + j] = acc;"),
    "A_transposed": (
        "acc += ad[i * K + k] * wrow[k];",
        "acc += ad[(k * nrows + i) % (nrows * K)] * wrow[k];"),
    "act_rows_transposed": (
        "ad[i * K + k] = act_value(A, a_is_bf16, m * K + k);",
        "ad[i * K + k] = act_value(A, a_is_bf16, (k * M + m) % (M * K));"),
    "fp8_A_transposed": (
        "acc += a8[k] * wrow[k];",
        "acc += ad[(k * nrows + i) % (nrows * K)] * wrow[k];"),
    "fp4_A_transposed": (
        "acc += a4[k] * wrow[k];",
        "acc += ad[(k * nrows + i) % (nrows * K)] * wrow[k];"),
    "round_ties_away": (
        "if (diff > 0.5 || (diff == 0.5 && fmod(fl, 2.0) != 0.0))",
        "if (diff >= 0.5)"),
    "f16_subnormal_scale": (
        "v = ldexp((double)m, -24);                 /* subnormal: m * 2^-24 */",
        "v = ldexp((double)m, -25);                 /* subnormal: m * 2^-24 */"),
    "quant_divisor": (
        "oracle_round_f16((double)(amax32 / 7.0f));",
        "oracle_round_f16((double)(amax32 / 8.0f));"),
    "quant_round_half_up": (
        "q = (int)rintf(x) + 8;",
        "q = (int)floorf(x + 0.5f) + 8;"),
    "quant_offset": (
        "q = (int)rintf(x) + 8;",
        "q = (int)rintf(x) + 7;"),
    "quant_scale_layout": (
        "s[g * N + n] = sb;",
        "s[n * (K / G) + g] = sb;"),
    "quant_nibble_order": (
        "w[n * (K / 2) + k / 2] |= (uint8_t)((k % 2 == 0) ? q : (q << 4));",
        "w[n * (K / 2) + k / 2] |= (uint8_t)((k % 2 == 1) ? q : (q << 4));"),
    "zp_index_transposed": (
        "int zero = z[grp * N + n];",
        "int zero = z[n * (K / G) + grp];"),
    "zp_A_transposed": (
        "dot += wrow[k] * arow[k];",
        "dot += wrow[k] * ad[(k * nrows + i) % (nrows * K)];"),
    "zp_ignored": (
        "return (double)(q - zero) * scale;",
        "return (double)(q - 8) * scale;"),
    "lut_index_reversed": (
        "double entry = oracle_f16_to_double(lut[code]);",
        "double entry = oracle_f16_to_double(lut[15 - code]);"),
    "lut_scale_dropped": (
        "    return entry * scale;",
        "    return entry;"),
    "lut_scale_transposed": (
        "double scale = oracle_f16_to_double(s[(k / G) * N + n]);\n    return entry * scale;",
        "double scale = oracle_f16_to_double(s[n * (K / G) + k / G]);\n    return entry * scale;"),
    "lut_A_transposed": (
        "sum += ad[K * i + k] * wv[k];",
        "sum += ad[(k * nrows + i) % (nrows * K)] * wv[k];"),
    "int2_offset": (
        "return (double)(q - 2) * scale;",
        "return (double)(q - 1) * scale;"),
    "int2_code_order": (
        "return (byte >> (2 * (k % 4))) & 0x3;",
        "return (byte >> (2 * (3 - k % 4))) & 0x3;"),
    "int2_pack_order": (
        "byte |= (uint8_t)((q[n * K + 4 * j + i] & 0x3) << (2 * i));",
        "byte |= (uint8_t)((q[n * K + 4 * j + i] & 0x3) << (6 - 2 * i));"),
    "int2_group_of_k": (
        "double scale = oracle_f16_to_double(s[(k / G) * N + n]);\n    return (double)(q - 2) * scale;",
        "double scale = oracle_f16_to_double(s[(k % (K / G)) * N + n]);\n    return (double)(q - 2) * scale;"),
    "int2_A_transposed": (
        "total += wv[k] * xa[k];",
        "total += wv[k] * ad[(k * nrows + i) % (nrows * K)];"),
    "pack_nibbles_swapped": (
        "w[n * (K / 2) + j] = (uint8_t)(lo | (hi << 4));",
        "w[n * (K / 2) + j] = (uint8_t)(hi | (lo << 4));"),
}


def _run_mutant(name, tmpdir):
    old, new = MUTATIONS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation {name}: pattern must occur exactly once"
    d = os.path.join(tmpdir, name)
    os.makedirs(d, exist_ok=True)
    c_path = os.path.join(d, "oracle.c")
    with open(c_path, "w") as f:
        f.write(src.replace(old, new))
    so = os.path.join(d, "liboracle_mutant.so")
    subprocess.run(["gcc", "-O2", "-fPIC", "-shared", "-ffp-contract=off", c_path, "-o", so, "-lm"],
                   check=True, capture_output=True)
    env = dict(os.environ, ORACLE_LIB=so)
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    return r.returncode


def test_every_planted_mistake_is_caught(tmp_path):
    names = sorted(MUTATIONS)
    with ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 1)) as ex:
        codes = list(ex.map(lambda n: _run_mutant(n, str(tmp_path)), names))
    survivors = [n for n, rc in zip(names, codes) if rc == 0]
    assert not survivors, f"mutations not caught by the pins: {survivors}"


def test_unmutated_copy_passes(tmp_path):
    # the harness itself: an unaltered copy built the same way passes the pins
    d = tmp_path / "clean"
    d.mkdir()
    shutil.copy(SRC, d / "oracle.c")
    so = str(d / "liboracle_clean.so")
    subprocess.run(["gcc", "-O2", "-fPIC", "-shared", "-ffp-contract=off", str(d / "oracle.c"), "-o", so,
                    "-lm"], check=True, capture_output=True)
    env = dict(os.environ, ORACLE_LIB=so)
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-2000:]
