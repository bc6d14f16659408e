"""bench.py's DRAM-traffic lookup on CPU: the table's lines are keyed by a hash of the kernel's
device code and headers without comments and blank lines, so that a comment edit keeps a capture
of the same code and any change of code retires it (the bench then reports no traffic)."""
import os
import shutil
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_code_only_drops_comments_and_blank_lines():
    src = "int a; // one\n\n/* two\n three */ int b;\n   // four\nint c;  \n"
    assert bench._code_only(src) == "int a;\n int b;\nint c;"


def _tree(tmp_path):
    root = tmp_path / "tree"
    csrc = root / "mixed_lora_projection_gb300" / "csrc"
    csrc.mkdir(parents=True)
    for f in ("kernels.cu", "kernels_w4.cu", "dev_common.cuh", "lora_internal.h", "lora_w4.h"):
        shutil.copy(os.path.join(ROOT, "mixed_lora_projection_gb300", "csrc", f), csrc / f)
    return root, csrc


def test_kernel_hash_ignores_comments_but_not_code(tmp_path, monkeypatch):
    root, csrc = _tree(tmp_path)
    monkeypatch.setattr(bench, "ROOT", str(root))
    h0, w0 = bench._kernel_hash(), bench._kernel_hash(True)
    k = csrc / "kernels.cu"
    text = k.read_text()
    # a comment and a blank line added inside the device part: the same hashes
    k.write_text(text.replace("namespace dev {", "namespace dev {\n// a note\n\n", 1))
    assert bench._kernel_hash() == h0 and bench._kernel_hash(True) == w0
    # a changed constant in the device part: a new bf16 hash
    k.write_text(text.replace("namespace dev {", "namespace dev {\nconstexpr int kProbe = 1;", 1))
    assert bench._kernel_hash() != h0
    # the shared header feeds both kernels' hashes
    k.write_text(text)
    hdr = csrc / "lora_internal.h"
    hdr.write_text(hdr.read_text() + "\nconstexpr int kProbe2 = 2;\n")
    assert bench._kernel_hash() != h0 and bench._kernel_hash(True) != w0

