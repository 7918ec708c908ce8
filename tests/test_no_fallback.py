"""The product path has no CPU fallback: the named ops refuse host tensors
(they never compute on the CPU), and nothing in the package imports the
oracle, which is test infrastructure.  CPU only."""
import ast
import os

import pytest
import torch

import fake_quant_numerics_gb300 as fq

PKG = os.path.dirname(fq.__file__)


@pytest.mark.parametrize("call", [
    lambda x: fq.fake_quant_int(x, 8, "symmetric", "tensor"),
    lambda x: fq.fake_quant_int(x.view(4, 64), 4, "affine", "row"),
    lambda x: fq.fake_quant_int(x.view(4, 64), 4, "symmetric", "group", group=32),
    lambda x: fq.fake_quant_fp8(x, "e5m2"),
    lambda x: fq.fake_quant_int_percentile(x, 8, "symmetric", 0.01),
    lambda x: fq.fake_quant_block(x, "e2m1", 16, "e4m3"),
    lambda x: fq.quantize_4bit_double(x),
])
def test_named_ops_refuse_host_tensors(call):
    x = torch.linspace(-1.0, 1.0, 256)
    with pytest.raises(ValueError, match="CUDA tensors only"):
        call(x)


def test_package_never_imports_the_oracle():
    for root, _, files in os.walk(PKG):
        for f in files:
            if not f.endswith(".py"):
                continue
            tree = ast.parse(open(os.path.join(root, f)).read())
            for node in ast.walk(tree):
                if isinstance(node, ast.Import):
                    names = [a.name for a in node.names]
                elif isinstance(node, ast.ImportFrom):
                    names = [node.module or ""]
                else:
                    continue
                assert not any(n == "oracle" or n.startswith("oracle.") for n in names), (f, names)
