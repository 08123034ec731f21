"""kernel_hash: what a profile's traffic figure is tied to.  It follows the
code of a kernel's translation unit and of the library headers it includes,
and ignores comments and layout, so documenting a header does not orphan the
measured profiles while any change of code does."""
import shutil

import pytest

from fsdp_emulated_ranks_gb300 import build as B


def test_code_tokens_drop_comments_and_keep_literals():
    src = ('int a = 1; // note\n/* block\n   comment */ const char* s = "x // y /* z */";\n'
           "#define X  2\nchar q = '\"';   int   b;\n")
    assert B.code_tokens(src) == ('int a = 1;\nconst char* s = "x // y /* z */";\n'
                                  "#define X 2\nchar q = '\"'; int b;")


@pytest.fixture
def tree(tmp_path, monkeypatch):
    """A copy of csrc/ and include/ that the test may edit."""
    csrc, inc = tmp_path / "csrc", tmp_path / "include"
    shutil.copytree(B.CSRC, csrc)
    shutil.copytree(B.INCLUDE, inc)
    monkeypatch.setattr(B, "CSRC", str(csrc))
    monkeypatch.setattr(B, "INCLUDE", str(inc))
    return csrc, inc


def test_hash_ignores_comments_but_not_code(tree):
    csrc, inc = tree
    before = B.kernel_hash("k_collectives.cu")
    header = inc / "cr.h"
    text = header.read_text()
    header.write_text(text.replace("#ifndef CR_H", "/* a new remark */\n#ifndef CR_H", 1))
    assert B.kernel_hash("k_collectives.cu") == before
    header.write_text(text.replace("#define CR_MAX_RANKS 64", "#define CR_MAX_RANKS 32", 1))
    assert B.kernel_hash("k_collectives.cu") != before
    header.write_text(text)
    fold = csrc / "fold.cuh"
    fold.write_text(fold.read_text() + "\nnamespace cr { inline int unused_probe() { return 1; } }\n")
    assert B.kernel_hash("k_collectives.cu") != before
