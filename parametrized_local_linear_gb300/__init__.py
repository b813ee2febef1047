"""GB300-native Parallax (parametrized local linear attention) forward."""
