"""The timeline debugging module's command line without a GPU: unknown or
missing arguments print the usage and return 2, before touching CUDA."""
from tensor_model_transformer_tp_gb300 import timeline


def test_usage_without_arguments(capsys):
    assert timeline.main([]) == 2
    assert "attn_bwd" in capsys.readouterr().out
    assert timeline.main(["gemm", "1"]) == 2
