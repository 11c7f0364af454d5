"""Without its compiled library the package refuses to run: there is no CPU
or Python fallback for the clip."""
import pytest

from global_l2_norm_gb300 import _abi


def test_missing_library_raises(monkeypatch, tmp_path):
    monkeypatch.setattr(_abi, "_LIB", None)
    monkeypatch.setattr(_abi, "lib_path", lambda: str(tmp_path / "libgclip.so"))
    with pytest.raises(RuntimeError, match="no fallback"):
        _abi.load()


def test_product_package_does_not_import_the_oracle():
    import ast
    import os
    root = os.path.dirname(_abi.__file__)
    for name in os.listdir(root):
        if name.endswith(".py"):
            tree = ast.parse(open(os.path.join(root, name)).read())
            for node in ast.walk(tree):
                if isinstance(node, (ast.Import, ast.ImportFrom)):
                    mods = [a.name for a in node.names] if isinstance(node, ast.Import) else [node.module or ""]
                    assert not any(m.split(".")[0] == "oracle" for m in mods), name
