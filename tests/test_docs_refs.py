"""Every file the design notes, the README and the profile summaries cite
by name exists in the repository (no GPU)."""
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SEARCH = ["", "long_context_mask_gb300", "long_context_mask_gb300/csrc", "tests", "tests/golden", "oracle",
          "include", "profiles"]


def _docs():
    docs = ["DESIGN.md", "README.md"]
    docs += [os.path.join("profiles", f) for f in sorted(os.listdir(os.path.join(ROOT, "profiles")))
             if f.endswith(".md")]
    return docs


@pytest.mark.parametrize("doc", _docs())
def test_cited_files_exist(doc):
    text = open(os.path.join(ROOT, doc), encoding="utf-8").read()
    missing = []
    for tok in re.findall(r"`([^`\s]+)`", text):
        if not re.search(r"\.(py|cu|cuh|h|c|cpp|md|txt|json)$", tok) or "*" in tok:
            continue
        if not any(os.path.exists(os.path.join(ROOT, d, tok)) for d in SEARCH):
            missing.append(tok)
    assert not missing, f"{doc} cites missing files: {missing}"
