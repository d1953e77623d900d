"""The C-ABI library loads and exports every entry point its header declares
(no GPU needed: nothing here launches work)."""
import ctypes
import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ts_sampler.h")


def declared_functions():
    text = open(HEADER, encoding="utf-8").read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ts_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for want in ("ts_create", "ts_destroy", "ts_sample", "ts_sample_debug", "ts_advance_steps",
                 "ts_read_status", "ts_status_string"):
        assert want in names


def test_library_exports_every_declared_symbol():
    import codebook_token_sampling_gb300 as ts
    lib = ctypes.CDLL(ts.LIB_PATH)
    for name in declared_functions():
        assert hasattr(lib, name), name
    assert set(ts.EXPORTED) == set(declared_functions())


def test_binding_exposes_c_names_and_constants():
    import codebook_token_sampling_gb300 as ts
    for name in declared_functions():
        assert callable(getattr(ts, name)), name
    text = open(HEADER, encoding="utf-8").read()
    for macro, value in re.findall(r"#define (TS_[A-Z0-9_]+) (\d+)u?", text):
        assert getattr(ts, macro) == int(value), macro
    assert ts.ts_status_string(ts.TS_OK) == "ok"
    assert ts.ts_status_string(ts.TS_ERR_UNSUPPORTED) == "unsupported size"


def test_status_codes_match_the_oracle_bits():
    import codebook_token_sampling_gb300 as ts
    import oracle
    assert (ts.TS_ROW_BAD_SHAPE, ts.TS_ROW_BAD_PARAM, ts.TS_ROW_NONFINITE, ts.TS_ROW_BAD_SLOT) == \
        (oracle.ERR_BAD_SHAPE, oracle.ERR_BAD_PARAM, oracle.ERR_NONFINITE, oracle.ERR_BAD_SLOT)


def _c_layout(tmp_path, struct, fields):
    """Offsets of `fields` in the header's `struct`, then its size, from a C
    program compiled against the header (gcc, no GPU)."""
    import subprocess
    body = "".join(f'printf("%zu\\n", offsetof({struct}, {f}));' for f in fields)
    src = tmp_path / f"{struct}.c"
    src.write_text('#include <stdio.h>\n#include <stddef.h>\n#include "ts_sampler.h"\n'
                   f'int main(void) {{ {body} printf("%zu\\n", sizeof({struct})); return 0; }}\n')
    exe = tmp_path / struct
    subprocess.run(["gcc", "-std=c11", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)],
                   check=True, capture_output=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout
    return [int(x) for x in out.split()]


def test_binding_structs_match_the_header(tmp_path):
    """Every field of the binding's ts_batch, ts_steps and ts_lm_head mirrors
    sits at the header's offset, and the sizes agree (a field missing, added
    or moved on either side fails here)."""
    import codebook_token_sampling_gb300 as ts
    for struct, mirror in (("ts_batch", ts.TsBatch), ("ts_steps", ts.TsSteps),
                           ("ts_lm_head", ts.TsLmHead)):
        fields = [name for name, _ in mirror._fields_]
        want = [getattr(mirror, f).offset for f in fields] + [ctypes.sizeof(mirror)]
        assert _c_layout(tmp_path, struct, fields) == want, struct
